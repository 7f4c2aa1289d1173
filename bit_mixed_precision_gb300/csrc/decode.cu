// decode_attn_qkv: one decode step of attention over the compressed cache,
// dequantising packed codes inside the kernel (MiKV rebuttal, the INTn x
// FP16 GEMV paragraph: on-the-fly dequantisation; MiniKV verdict JSON
// forward_implications: fused dequantisation kernels during decoding).
//
// One launch per step.  Each (batch, KV head) unit is one thread-block
// cluster of C CTAs (C = 1 .. 16: as many as one wave holds for small
// caches, fewer for large ones).  The unit's work is a list of items:
// 128-token sub-chunks of every packed tier, then 8-row pieces of the
// residual ring (the new token last); the CTA of item rank q takes items
// q, q + C, q + 2C, ... (the leader has the last rank).  A CTA requests
// each item with bulk asynchronous copies into one of S staging buffers
// (S = 2 or 4; item i + S is requested as soon as every warp is done with
// item i); its four warps take 32 tokens (or 2 residual rows) each: keys ->
// base-2 logits for the g query heads of the KV head (tensor cores for
// head dim 128), online softmax per warp, P.V with the codes turned into
// fp16 by one rotate or byte permute and one LOP3 per pair.  The CTA merges
// its warps and writes its partial (max, sum, unnormalised output) into
// the shared memory of the cluster's leader (distributed shared memory, no
// global round trip, no atomics).  The leader merges the C partials and
// writes o and lse.  Then, per policy:
//   DiffKV / MiKV: the leader broadcasts the log-sum-exp and every CTA adds
//     this step's attention to the scores of its own tokens (DiffKV: per
//     ring slot and query head; MiKV: per token, summed over the group);
//   MiniKV: when the residual reaches nr + G tokens the leader packs its G
//     oldest into tier 0 (MiniKV review, nr; verdict JSON key_machinery).
// The new token joins the ring at the start (from the cluster's last CTA;
// its slot is not read this step) and the leader advances res_len and the
// unit's position at the end.  Tiers are read where they lie (MiKV rebuttal:
// attention is permutation invariant, so each precision group sits in its
// own region).
#include <algorithm>
#include <atomic>
#include <mutex>

#include "kvq_common.cuh"
#include "kvq_internal.h"
#include "pack_device.cuh"

namespace kvq {

KVQ_DEFINE_STATUS(decode)

namespace {

constexpr int kSub = 128;        // packed tokens per item, split evenly over the warps
constexpr int kResItem = 8;      // residual rows per item (small: the fp16 rows are the heaviest bytes)
constexpr int kMaxCluster = 16;
constexpr int kMaxStages = 4;    // staging buffers per CTA (2 or 4)
constexpr uint32_t kSleepNs = 4000;  // longest single suspension of a waiting warp
// large caches: items a CTA streams at least (measured per workload: the MiKV cache, two
// per-token tiers behind a 32k prompt, runs 7 % faster at C = 4 than at C = 8, i.e. with
// about twice as many items per CTA as the others want)
constexpr int kMinItemsPerCta = 34, kMinItemsPerCtaMikv = 64;
// streamed decode: CTAs at most (the workspace holds one partial per (CTA, unit) pair, at
// most ctas + units - 1 of them), and static items per CTA at least
constexpr int kStreamMaxCtas = 1024, kStreamMinItems = 8;
// streamed decode: residual rows per ring item (eight per warp: fewer items per unit than the
// cluster path's 8-row pieces, which spread the ring over the cluster's CTAs)
constexpr int kResItemS = 32;
// streamed decode: tier chunk tokens (256 where two buffers of them keep four CTAs per SM)
template <int GK>
constexpr int kStreamChunk = GK == 32 ? 256 : 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kNegInf = -__builtin_huge_valf();

// Four warps per CTA, 32 packed tokens each per item.
template <int NG>
struct Cfg {
    static constexpr int W = 4;
    static constexpr int kThreads = W * 32;
    static constexpr int TPW = kSub / W;        // packed tokens per warp and item
    static constexpr int REP = 32 / TPW;        // lanes holding one token's logit
    static constexpr int RPW = kResItem / W;    // residual rows per warp and item
    static constexpr int MINB = NG == 1 ? 4 : (NG <= 4 ? 3 : 2); // resident CTAs per SM the registers must allow
};

struct TierArgs {
    int k_bits, v_bits, k_axis, cap;
    uint32_t* k_codes;
    uint16_t* k_scale;
    uint16_t* k_zero;
    uint32_t* v_codes;
    uint16_t* v_scale;
    uint16_t* v_zero;
    int32_t* token_id;
    int32_t* count;
    int slot_base;              // offset of this tier in the logits row
    const int32_t* page_table;  // paged tier: [unit][max_pages] physical page of each 128-slot chunk
    int max_pages, n_pages;
};

struct DecodeArgs {
    const void* q;
    const void* k_new;
    const void* v_new;
    void* o;
    float* lse_out;
    int B, Hq, Hkv, D, G, g, n_tiers, policy, bf16, nr;
    TierArgs tier[KVQ_MAX_TIERS];
    void* res_k;
    void* res_v;
    int32_t* res_token_id;
    int32_t* res_start;
    int32_t* res_len;
    int res_cap, res_slot_base;
    int32_t* pos;               // [units] position of the next token
    float* win_acc;
    float* cum_score;
    int score_cap;
    float scale_log2;
    int slots;                  // logits row length per (unit, head)
    float* logits;              // [unit][g][slots] (DiffKV, MiKV) or null
    float* lse2_ws;             // MiKV: [unit][8] the step's base-2 lse per head, for the score kernel
    int32_t* meta_ws;           // MiKV: [unit][4] ring length, first slot and position before the step
    int cluster;                // CTAs per unit
    uint32_t stage_bytes;       // one staging buffer
    int stages, stage_shift;    // staging buffers per CTA (2 or 4) and its log2
    int withhold_unit;          // failure-detection check: unit whose first CTA skips its first copy, or -1
    uint32_t qf_off, part_off, stage_off;  // dynamic shared memory offsets
    float* stream_part;         // streamed decode: partial per (CTA, unit), in the workspace
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

// 32 lanes each hold v[0..N-1] (N = 4 .. 32); afterwards the 32/N lanes
// (32/N) t .. (32/N) t + 32/N - 1 return the sum over lanes of v[t].
template <int N>
__device__ __forceinline__ float reduce_scatter(float (&v)[N]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int half = N / 2, s = 16; half >= 1; half >>= 1, s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = up ? v[i] : v[i + half];
            const float keep = up ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
#pragma unroll
    for (int s = 16 / N; s >= 1; s >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], s);
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

// Per-unit state read once at the start of the launch (before any CTA of
// the cluster can change it) and the item map derived from it.
struct UnitState {
    int cnt[KVQ_MAX_TIERS];              // valid slots of each tier
    int base[KVQ_MAX_TIERS + 1];         // first item of each tier; base[n_tiers] = first residual item
    int len, start, pos;                 // residual length and first slot, position of the new token
    int total;                           // items of the unit
};

template <int NG, int D>
struct Smem {
    float q[NG][D];                      // query rows, pre-scaled to base-2 logits
    float wm[Cfg<NG>::W][NG];            // per-warp running max / sum / output (merged across kinds)
    float wl[Cfg<NG>::W][NG];
    float wo[Cfg<NG>::W][NG][D];
    // logits of the warp's current group (CUDA-core per-token path: single heads only)
    // (single heads, MiniKV format: the warp's probabilities, 32 floats, then in the same
    // bytes the probabilities times each value group's scale, fp16 [group][40: 32 tokens])
    float lg[NG == 1 ? Cfg<NG>::W : 1][1][NG == 1 ? 80 : 1];
    // per-token keys (GQA groups): the query's A fragments, [k-step][lane] (single heads: unused)
    uint4 qa[NG >= 2 ? 8 : 1][32];
    float cw[kMaxCluster][NG];           // leader: weight of each CTA partial
    float lse2[NG];                      // base-2 log-sum-exp of the step (broadcast by the leader)
    float lsum[NG];
    unsigned long long bar[kMaxStages];  // one staging mbarrier per buffer
    int issued;                          // local items requested so far (thread 0 requests)
    int fail;                            // a wait gave up: nothing more is requested
    UnitState us;
    // streamed decode: the item of each buffer (unit, kind, index, tokens), and the issuing
    // thread's cursor (next static item, its unit's counters, whether that unit has an item)
    int4 meta[kMaxStages];
    int wu, wk, wrem;
    int cu, ccnt, clen, cstart, cem;
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

// Logits of the warp's tokens (lanes REP t .. REP t + REP - 1 hold token t;
// tokens from nt on are absent) -> rescale the accumulators, return p_h(t)
// in lg and write the logits out when asked.
template <int REP, int NG, int NO>
__device__ __forceinline__ void group_softmax(WarpAcc<NG, NO>& acc, float (&lg)[NG], int nt,
                                              float* lg_out, int slots) {
    const int lane = threadIdx.x & 31;
    const int tok = lane / REP;
    const bool lead = lane % REP == 0, valid = tok < nt;
#pragma unroll
    for (int h = 0; h < NG; ++h) {
        const float s = valid ? lg[h] : kNegInf;
        if (lg_out && valid && lead) lg_out[(size_t)h * slots + tok] = s;
        const float mn = fmaxf(acc.m[h], warp_max(s));
        const float corr = acc.m[h] == kNegInf ? 0.0f : ex2_approx(acc.m[h] - mn);
        const float p = valid ? ex2_approx(s - mn) : 0.0f;
        acc.l[h] = acc.l[h] * corr + warp_sum(lead ? p : 0.0f);
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

__device__ __forceinline__ View view_of(const StageSizes& z, const uint8_t* buf);

__device__ __forceinline__ View tier_view(const TierArgs& t, int npad, int D, int G, const uint8_t* buf) {
    return view_of(tier_stage_sizes(t.k_axis, t.k_bits, t.v_bits, npad, D, G), buf);
}

// The same view for a format known at compile time (D = 128, G = 32: the
// sizes fold to shifts of npad).
template <int KB, int KAX, int VB>
__device__ __forceinline__ View tier_view_c(int npad, const uint8_t* buf) {
    return view_of(tier_stage_sizes(KAX, KB, VB, npad, 128, 32), buf);
}

__device__ __forceinline__ View view_of(const StageSizes& z, const uint8_t* buf) {
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

// The six arrays of tokens [j0, j0 + npad) of a tier: fn(global source,
// bytes, offset in the staged chunk) for each.
template <typename Fn>
__device__ __forceinline__ void tier_ranges(const TierArgs& t, size_t unit, int j0, int npad, int D, int G,
                                            Fn fn) {
    const StageSizes z = tier_stage_sizes(t.k_axis, t.k_bits, t.v_bits, npad, D, G);
    // a paged tier's chunk (128 slots) is one page: the page's rows stand in for the unit's
    size_t urow = unit;
    int cap = t.cap;
    if (t.page_table) {
        int pg = t.page_table[unit * (size_t)t.max_pages + j0 / KVQ_PAGE_TOKENS];
        if (pg < 0 || pg >= t.n_pages) {
            atomicOr(&g_status_decode, kDevCheck);
            pg = 0;
        }
        urow = (size_t)pg;
        j0 -= (j0 / KVQ_PAGE_TOKENS) * KVQ_PAGE_TOKENS;
        cap = KVQ_PAGE_TOKENS;
    }
    const void *kc_src, *ks_src, *kz_src;
    if (t.k_axis == KVQ_AXIS_CHANNEL) {
        const int per = 32 / t.k_bits;
        kc_src = t.k_codes + (urow * (size_t)(cap / per) + j0 / per) * D;
        const size_t so = (urow * (size_t)(cap / G) + j0 / G) * D;
        ks_src = t.k_scale + so;
        kz_src = t.k_zero + so;
    } else {
        kc_src = t.k_codes + (urow * (size_t)cap + j0) * (D * t.k_bits / 32);
        const size_t so = (urow * (size_t)cap + j0) * (D / G);
        ks_src = t.k_scale + so;
        kz_src = t.k_zero + so;
    }
    const size_t vo = urow * (size_t)cap + j0;
    const uint32_t o_ks = a16(z.kc), o_kz = o_ks + a16(z.ks), o_vc = o_kz + a16(z.ks);
    const uint32_t o_vs = o_vc + a16(z.vc), o_vz = o_vs + a16(z.vs);
    fn(kc_src, z.kc, 0u);
    fn(ks_src, z.ks, o_ks);
    fn(kz_src, z.ks, o_kz);
    fn(t.v_codes + vo * (D * t.v_bits / 32), z.vc, o_vc);
    fn(t.v_scale + vo * (D / G), z.vs, o_vs);
    fn(t.v_zero + vo * (D / G), z.vs, o_vz);
}

// Called by one thread: the six bulk copies of tokens [j0, j0 + npad) of a tier.
__device__ void stage_tier(const TierArgs& t, size_t unit, int j0, int npad, int D, int G,
                           const uint8_t* buf, uint32_t bar) {
    const StageSizes z = tier_stage_sizes(t.k_axis, t.k_bits, t.v_bits, npad, D, G);
    const uint32_t d = smem_u32(buf);
    mbar_expect_tx(bar, z.kc + 2 * z.ks + z.vc + 2 * z.vs);
    tier_ranges(t, unit, j0, npad, D, G,
                [&](const void* src, uint32_t bytes, uint32_t off) { bulk_load(d + off, src, bytes, bar); });
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
    constexpr int TPW = Cfg<NG>::TPW;
    constexpr int per = 32 / KB;          // tokens per word
    constexpr int rows = TPW / per;       // word rows per warp
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
        float part[TPW];
#pragma unroll
        for (int k = 0; k < TPW; ++k) part[k] = 0.0f;
#pragma unroll
        for (int r = 0; r < rows; ++r)
#pragma unroll
            for (int ci = 0; ci < CPL; ++ci)
#pragma unroll
                for (int i = 0; i < per; ++i)
                    part[r * per + i] = fmaf(code_f<KB>(w[r][ci], i), qs[ci], part[r * per + i]);
        const float raw = reduce_scatter<TPW>(part);
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
    for (int ps = 0; ps < Cfg<NG>::TPW / tpp; ++ps) {
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
    for (int h = 0; h < NG; ++h) lg[h] = sm.lg[warp][h][lane / Cfg<NG>::REP];
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
    for (int ps = 0; ps < Cfg<NG>::TPW / tpp; ++ps) {
        const int tk = ps * tpp + to;
        float pk[NG];
#pragma unroll
        for (int h = 0; h < NG; ++h) pk[h] = __shfl_sync(0xffffffffu, p[h], tk * Cfg<NG>::REP);
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

// ---- merging a warp's register state into its shared-memory state

// Combines the warp's (m, l) with the stored ones; returns the factors that
// scale the stored and the new output.  m and l are uniform over the warp.
template <int NG, int D, int NO>
__device__ __forceinline__ void merge_stats(Smem<NG, D>& sm, const WarpAcc<NG, NO>& acc,
                                            float (&fo)[NG], float (&fn)[NG]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float M[NG], L[NG];
#pragma unroll
    for (int h = 0; h < NG; ++h) {
        const float mo = sm.wm[warp][h];
        M[h] = fmaxf(mo, acc.m[h]);
        fo[h] = mo == kNegInf ? 0.0f : ex2_approx(mo - M[h]);
        fn[h] = acc.m[h] == kNegInf ? 0.0f : ex2_approx(acc.m[h] - M[h]);
        L[h] = sm.wl[warp][h] * fo[h] + acc.l[h] * fn[h];
    }
    __syncwarp();
    if (lane == 0) {
#pragma unroll
        for (int h = 0; h < NG; ++h) {
            sm.wm[warp][h] = M[h];
            sm.wl[warp][h] = L[h];
        }
    }
}

// Packed-V layout: remove the constants, sum the lanes that share a word,
// merge into the warp's output.
template <int VB, int D, int NG>
__device__ __forceinline__ void flush_token_values(WarpAcc<NG, 32 / VB>& acc, Smem<NG, D>& sm) {
    constexpr int lpt = D * VB / 32, cpw = 32 / VB;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int wi = lane % lpt, to = lane / lpt;
    float fo[NG], fn[NG];
    merge_stats(sm, acc, fo, fn);
#pragma unroll
    for (int h = 0; h < NG; ++h)
#pragma unroll
        for (int i = 0; i < cpw; ++i) {
            float x = (acc.o[h][i] - acc.off[h]) * (float)(1 << VB) + acc.zs[h];
#pragma unroll
            for (int o = lpt; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
            if (to == 0) {
                float* p = &sm.wo[warp][h][wi * cpw + i];
                *p = *p * fo[h] + x * fn[h];
            }
        }
    __syncwarp();
}

// Residual layout: lane owns channels [lane * CPL, lane * CPL + CPL).
template <int NG, int D>
__device__ __forceinline__ void flush_lane_values(WarpAcc<NG, D / 32>& acc, Smem<NG, D>& sm) {
    constexpr int CPL = D / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float fo[NG], fn[NG];
    merge_stats(sm, acc, fo, fn);
#pragma unroll
    for (int h = 0; h < NG; ++h)
#pragma unroll
        for (int ci = 0; ci < CPL; ++ci) {
            float* p = &sm.wo[warp][h][lane * CPL + ci];
            *p = *p * fo[h] + acc.o[h][ci] * fn[h];
        }
    __syncwarp();
}

// ---- residual rows (full precision), eight per warp

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

// Rows [0, nt) (nt <= RPW) of the warp's slice: logits, online softmax and
// P.V; the logits go to lg_out (row-indexed) when asked.
template <int NG, int D, int RPW = Cfg<NG>::RPW>
__device__ __forceinline__ void residual_rows(const Smem<NG, D>& sm, const uint16_t* rk,
                                              const uint16_t* rv, int nt, bool bf,
                                              WarpAcc<NG, D / 32>& acc, float* lg_out, int slots) {
    constexpr int CPL = D / 32;
    constexpr int LPR = 32 / RPW;                  // lanes per row (RPW rows per warp)
    const int lane = threadIdx.x & 31;
    const int c0 = lane * CPL;
    const int t = lane / LPR;                      // the row this lane reports
    float lg[NG];
#pragma unroll 1
    for (int h = 0; h < NG; ++h) {
        float part[RPW];
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
            part[k] = 0.0f;
            if (k < nt) {
                float x[CPL];
                row_vals<CPL>(rk + (size_t)k * D + c0, bf, x);
#pragma unroll
                for (int ci = 0; ci < CPL; ++ci) part[k] = fmaf(sm.q[h][c0 + ci], x[ci], part[k]);
            }
        }
        lg[h] = reduce_scatter<RPW>(part);
    }
    const bool valid = t < nt, lead = lane % LPR == 0;
#pragma unroll
    for (int h = 0; h < NG; ++h) {
        const float s = valid ? lg[h] : kNegInf;
        if (lg_out && valid && lead) lg_out[(size_t)h * slots + t] = s;
        const float mn = fmaxf(acc.m[h], warp_max(s));
        const float corr = acc.m[h] == kNegInf ? 0.0f : ex2_approx(acc.m[h] - mn);
        const float p = valid ? ex2_approx(s - mn) : 0.0f;
        acc.l[h] = acc.l[h] * corr + warp_sum(lead ? p : 0.0f);
#pragma unroll
        for (int ci = 0; ci < CPL; ++ci) acc.o[h][ci] *= corr;
        acc.m[h] = mn;
        lg[h] = p;
    }
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
        if (k < nt) {
            float x[CPL];
            row_vals<CPL>(rv + (size_t)k * D + c0, bf, x);
#pragma unroll
            for (int h = 0; h < NG; ++h) {
                const float pk = __shfl_sync(0xffffffffu, lg[h], LPR * k);
#pragma unroll
                for (int ci = 0; ci < CPL; ++ci) acc.o[h][ci] = fmaf(pk, x[ci], acc.o[h][ci]);
            }
        }
    }
}

// ---- items

// Global item k of the unit: tier (or -1 for the residual) and index within it.
__device__ __forceinline__ int item_kind(const UnitState& us, int n_tiers, int k, int& idx) {
    for (int t = 0; t < n_tiers; ++t)
        if (k < us.base[t + 1]) {
            idx = k - us.base[t];
            return t;
        }
    idx = k - us.base[n_tiers];
    return -1;
}

// First local index of the CTA of item rank r (items r, r + C, ...) at or
// after global item k.  Item functions below take that rank as r.
__device__ __forceinline__ int local_at(int k, int r, int C) { return k > r ? (k - r + C - 1) / C : 0; }

// Called by one thread at the start, while another thread reads the unit's
// counters: L2 prefetches of what this CTA will most likely stage first (its
// first two sub-chunks of tier 0 at full capacity and a 1/C share of the
// residual ring), and of the new token's rows the leader appends at the end.
__device__ void prefetch_start(const DecodeArgs& a, size_t unit, int r) {
    const int C = a.cluster, D = a.D;
    const TierArgs& t0 = a.tier[0];
    const int nsub = t0.page_table ? 0 : (t0.cap + kSub - 1) / kSub;   // pages: unknown until read
    for (int k = r, i = 0; k < nsub && i < 2; k += C, ++i) {
        const int j0 = k * kSub;
        tier_ranges(t0, unit, j0, min(kSub, t0.cap - j0), D, a.G,
                    [&](const void* src, uint32_t bytes, uint32_t) {
                        if (bytes) bulk_prefetch_l2(src, bytes);
                    });
    }
    const int share = (a.res_cap + C - 1) / C, r0 = r * share, n = min(share, a.res_cap - r0);
    if (n > 0) {
        const uint32_t bytes = (uint32_t)n * D * 2;
        bulk_prefetch_l2(reinterpret_cast<const uint16_t*>(a.res_k) + (unit * a.res_cap + r0) * D, bytes);
        bulk_prefetch_l2(reinterpret_cast<const uint16_t*>(a.res_v) + (unit * a.res_cap + r0) * D, bytes);
    }
    if (r == 0) {
        bulk_prefetch_l2(reinterpret_cast<const uint16_t*>(a.k_new) + unit * D, (uint32_t)D * 2);
        bulk_prefetch_l2(reinterpret_cast<const uint16_t*>(a.v_new) + unit * D, (uint32_t)D * 2);
    }
}

// Called by one thread: the bulk copies of local item i into buffer i % S.
__device__ void issue_item(const DecodeArgs& a, const UnitState& us, size_t unit, int r, int i,
                           uint8_t* stage_base, const unsigned long long* bars) {
    const int D = a.D;
    int idx;
    const int t = item_kind(us, a.n_tiers, r + i * a.cluster, idx);
    const int sb = i & (a.stages - 1);
    uint8_t* buf = stage_base + (size_t)sb * a.stage_bytes;
    const uint32_t bar = smem_u32(&bars[sb]);
    if (t >= 0) {
        const int j0 = idx * kSub;
        const int n = min(kSub, us.cnt[t] - j0);
        stage_tier(a.tier[t], unit, j0, (n + 31) & ~31, D, a.G, buf, bar);
    } else {
        const int j0 = idx * kResItem;
        const int n = min(kResItem, us.len + 1 - j0);
        stage_residual(a, unit, us.len, us.start, j0, n, D, buf, bar);
    }
}

// Buffer of local item i.
__device__ __forceinline__ const uint8_t* item_buf(const DecodeArgs& a, const uint8_t* stage_base, int i) {
    return stage_base + (size_t)(i & (a.stages - 1)) * a.stage_bytes;
}

// Waits for local item i (buffer i % S, phase i / S).  Each warp waits on
// its own: lane 0 polls the mbarrier, suspended between tests (bounded, and
// cut short once another warp has given up), then every lane tests the
// completed phase once, which acquires the copied bytes.
template <int NG, int D>
__device__ __forceinline__ bool wait_item(const DecodeArgs& a, Smem<NG, D>& sm, int i, bool ok) {
    const uint32_t bar = smem_u32(&sm.bar[i & (a.stages - 1)]), par = (uint32_t)(i >> a.stage_shift) & 1u;
    const int lane = threadIdx.x & 31;
    int mine = ok ? 1 : 0;
    if (lane == 0 && ok) {
        mine = mbar_wait_sleep(bar, par, &sm.fail, kSleepNs) ? 1 : 0;
        if (!mine) *(volatile int*)&sm.fail = 1;
    }
    mine = __shfl_sync(0xffffffffu, mine, 0);
    if (mine) (void)mbar_try_wait(bar, par);
    return mine != 0;
}

// Every warp is done with local item i: thread 0 requests item i + S into
// the same buffer (nothing more once a wait has given up).
template <int NG, int D>
__device__ __forceinline__ void release_item(const DecodeArgs& a, Smem<NG, D>& sm, size_t unit, int r, int i,
                                             int n_local, uint8_t* stage_base) {
    __syncthreads();
    if (threadIdx.x == 0 && i + a.stages < n_local && !sm.fail) {
        issue_item(a, sm.us, unit, r, i + a.stages, stage_base, sm.bar);
        sm.issued = i + a.stages + 1;
    }
}

// Local items [i0, i1) of one packed tier.
template <int KB, int KAX, int VB, int D, int NG>
__device__ void run_tier(const DecodeArgs& a, Smem<NG, D>& sm, int t, size_t unit, int r, int i0,
                         int i1, int n_local, uint8_t* stage_base, float* lg_unit, bool& ok) {
    const TierArgs& ta = a.tier[t];
    const UnitState& us = sm.us;
    const int warp = threadIdx.x >> 5;
    constexpr int TPW = Cfg<NG>::TPW;
    WarpAcc<NG, 32 / VB> acc;
    acc_init(acc);
    for (int i = i0; i < i1; ++i) {
        ok = wait_item(a, sm, i, ok);
        if (ok) {
            const int j0 = (r + i * a.cluster - us.base[t]) * kSub;
            const int n = min(kSub, us.cnt[t] - j0);
            const View v = tier_view(ta, (n + 31) & ~31, D, a.G, item_buf(a, stage_base, i));
            const int tl = warp * TPW;
            if (tl < n) {
                const int nt = min(TPW, n - tl);
                float lg[NG];
                if constexpr (KAX == KVQ_AXIS_CHANNEL)
                    logits_channel<KB, D / 32, NG>(v, tl, sm, a.G, lg);
                else
                    logits_token<KB, D, NG>(v, tl, sm, a.G, lg);
                float* lo = (a.policy == KVQ_POLICY_MIKV && lg_unit) ? lg_unit + ta.slot_base + j0 + tl : nullptr;
                group_softmax<Cfg<NG>::REP>(acc, lg, nt, lo, a.slots);
                values_token<VB, D, NG>(v, tl, nt, lg, a.G, acc);
            }
        }
        release_item(a, sm, unit, r, i, n_local, stage_base);
    }
    flush_token_values<VB, D, NG>(acc, sm);
}

// ---- tensor-core path for per-token tiers (GQA groups, D = 128, G = 32)
//
// Each warp takes 32 tokens of an item.  Logits: mma.m16n8k16 with the
// query group as A (16 rows: row 2h holds head h's query rounded to fp16,
// row 2h + 1 the fp16 rounding remainder, so that the pair carries the
// float32 query) and the packed key codes as B, each code turned into the
// fp16 value 1 + c / 2^KB by one rotate and one LOP3 (two codes per 32-bit
// register).  The channels of a k-step are permuted so that both codes of
// a register come from one packed word; the query side uses the same
// permutation.  One accumulator per 32-channel group takes the token's
// scale and zero in float32 afterwards.  P.V: the probabilities (again a
// hi / lo row pair) are the A operand straight from the logit accumulators;
// B holds the value codes of two tokens per register (byte permute, shift,
// LOP3) times their fp16 scale (one fused multiply-add, one rounding); the
// zero points are summed per group in float32.

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two floats -> f16x2 (round to nearest), lo in the low half.
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ float h2lo(uint32_t x) { return __half2float(__ushort_as_half((unsigned short)(x & 0xffffu))); }
__device__ __forceinline__ float h2hi(uint32_t x) { return __half2float(__ushort_as_half((unsigned short)(x >> 16))); }

// Codes j and j + 16/KB of a packed word (bits KB*j and KB*j + 16) as the
// f16x2 pair (1 + c_j / 2^KB, 1 + c_{j+16/KB} / 2^KB).
template <int KB>
__device__ __forceinline__ uint32_t code_pair(uint32_t w, int j) {
    const int rot = ((10 - KB - KB * j) % 32 + 32) % 32;
    const uint32_t x = __funnelshift_l(w, w, rot);
    constexpr uint32_t m = ((1u << KB) - 1u) << (10 - KB);
    return (x & (m | (m << 16))) | 0x3C003C00u;
}

// Channels (lo, hi) of the register b (0: k 2t..2t+1, 1: k 2t+8..2t+9) of
// thread t in k-step s, and the word of the token row that holds them.
template <int KB>
__device__ __forceinline__ void kchan(int s, int t, int b, int& word, int& j, int& c_lo, int& c_hi) {
    const int grp = s >> 1, e = s & 1;
    if (KB == 4) {                       // word 4 grp + t, pairs (j, j + 4)
        word = 4 * grp + t;
        j = 2 * e + b;
        c_lo = 8 * word + j;
        c_hi = c_lo + 4;
    } else if (KB == 8) {                // words 8 grp + 2t + e, pairs (j, j + 2)
        word = 8 * grp + 2 * t + e;
        j = b;
        c_lo = 4 * word + j;
        c_hi = c_lo + 2;
    } else {                             // KB == 2: word 2 grp + t/2, pairs (j, j + 8)
        word = 2 * grp + (t >> 1);
        j = 4 * (t & 1) + 2 * e + b;
        c_lo = 16 * word + j;
        c_hi = c_lo + 8;
    }
}

template <int NG>
struct MmaAcc {
    static constexpr int RI = NG > 4 ? 2 : 1;   // blocks of 4 heads (8 hi / lo rows)
    float m[RI], l[RI];                          // logit layout: row g + 8 ri
    // P.V layout, D = V^T P: [16-channel m-tile][head block][channel g, g+8 x rows 2t, 2t+1],
    // i.e. this lane holds head 4 ri + t (hi and lo rows) for channels 16 mt + g and + 8
    float o[8][RI][4];
    float zs[RI][4];                             // sum of p * zero per value group (logit layout)
};

// Query fragments for the channel permutation of KB-bit keys, times 2^KB
// (exact: a power of two), and the per-group sums of each fragment row
// (without the factor).
template <int KB, int NG, int D>
__device__ __forceinline__ void build_qa(Smem<NG, D>& sm, float (&qs)[4][2]) {
    uint32_t qa[8][4];
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    auto part = [&](int row, int c) -> float {
        const int h = row >> 1;
        if (h >= NG) return 0.0f;
        const float x = sm.q[h][c] * (float)(1 << KB);
        const float hi = __half2float(__float2half_rn(x));
        return (row & 1) ? __half2float(__float2half_rn(x - hi)) : hi;
    };
#pragma unroll
    for (int grp = 0; grp < 4; ++grp) qs[grp][0] = qs[grp][1] = 0.0f;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            int word, j, c_lo, c_hi;
            kchan<KB>(s, t, b, word, j, c_lo, c_hi);
#pragma unroll
            for (int ri = 0; ri < 2; ++ri) {
                const int row = g + 8 * ri;
                const float x0 = part(row, c_lo), x1 = part(row, c_hi);
                qa[s][2 * b + ri] = pack_h2(x0, x1);
                qs[s >> 1][ri] += x0 + x1;
            }
        }
    }
#pragma unroll
    for (int grp = 0; grp < 4; ++grp)
#pragma unroll
        for (int ri = 0; ri < 2; ++ri) {
            qs[grp][ri] += __shfl_xor_sync(0xffffffffu, qs[grp][ri], 1);
            qs[grp][ri] += __shfl_xor_sync(0xffffffffu, qs[grp][ri], 2);
            qs[grp][ri] *= 1.0f / (float)(1 << KB);
        }
    if (threadIdx.x < 32)                                // every warp holds the same values
#pragma unroll
        for (int st = 0; st < 8; ++st) sm.qa[st][lane] = make_uint4(qa[st][0], qa[st][1], qa[st][2], qa[st][3]);
}

// Logits of the warp's 32 tokens, keys per token (KB bits):
// S[n-tile][rows g, g+8 x tokens 2t, 2t+1], hi and lo rows not yet summed.
template <int KB, int NG, int NT>
__device__ __forceinline__ void mma_logits_token(const View& v, int tl, const uint4 (&qa)[8][32],
                                                 const float (&qs)[4][2], float (&S)[NT][4]) {
    constexpr int D = 128, GR = 4;                       // channels, 32-channel groups
    constexpr int RI = MmaAcc<NG>::RI;
    constexpr int kw = D * KB / 32;                      // words per token row
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) S[n][i] = 0.0f;
#pragma unroll
    for (int grp = 0; grp < GR; ++grp) {
        float R[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
#pragma unroll
            for (int i = 0; i < 4; ++i) R[n][i] = 0.0f;
            const uint32_t* row = v.kc + (size_t)(tl + 8 * n + g) * kw;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                int w0, j0, c0, c1, w1, j1;
                kchan<KB>(2 * grp + e, t, 0, w0, j0, c0, c1);
                kchan<KB>(2 * grp + e, t, 1, w1, j1, c0, c1);
                const uint32_t b0 = code_pair<KB>(row[w0], j0);
                const uint32_t b1 = code_pair<KB>(row[w1], j1);
                const uint4 q4 = qa[2 * grp + e][lane];
                const uint32_t af[4] = {q4.x, q4.y, q4.z, q4.w};
                mma16816(R[n], af, b0, b1);
            }
        }
        // R carries the factor 2^KB of the fragments: s R = (2^KB s) R_1, and
        // zp = z - 2^KB s (both exact rewrites of the unscaled form).  The two
        // tokens 2t, 2t + 1 of a row go together, on packed float32 pairs.
        const unsigned long long mk2 = f2_pack(-(float)(1 << KB), -(float)(1 << KB));
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const int tok = tl + 8 * n + 2 * t;
            const unsigned long long s2 = f2_pack(h2f_bits(v.ks[tok * GR + grp]), h2f_bits(v.ks[(tok + 1) * GR + grp]));
            const unsigned long long zp2 =
                f2_fma(s2, mk2, f2_pack(h2f_bits(v.kz[tok * GR + grp]), h2f_bits(v.kz[(tok + 1) * GR + grp])));
#pragma unroll
            for (int ri = 0; ri < RI; ++ri) {
                unsigned long long a2 = f2_pack(S[n][2 * ri], S[n][2 * ri + 1]);
                a2 = f2_fma(f2_pack(qs[grp][ri], qs[grp][ri]), zp2, a2);
                a2 = f2_fma(s2, f2_pack(R[n][2 * ri], R[n][2 * ri + 1]), a2);
                f2_unpack(a2, S[n][2 * ri], S[n][2 * ri + 1]);
            }
        }
    }
}

// Logits of the warp's 32 tokens, keys per channel (INT2, one scale row for
// the 32 tokens): the query times the channel scales, as hi / lo fp16 rows,
// goes through the warp's shared rows qf (A operand); the codes of two
// channels of one token meet in one register by a byte permute.
template <int NG, int NT>
__device__ __forceinline__ void mma_logits_channel(const View& v, int tl, int G, const float (&q)[NG][128],
                                                   uint16_t (&qf)[2 * NG][128], float (&S)[NT][4]) {
    constexpr int D = 128;
    static_assert(NG <= 4, "rows g only");
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    // A rows for this scale row, and the per-row constants
    const uint16_t* ks = v.ks + (size_t)(tl / G) * D;
    const uint16_t* kz = v.kz + (size_t)(tl / G) * D;
    float cst[2 * NG];
#pragma unroll
    for (int h = 0; h < NG; ++h) {
        float shi = 0.0f, slo = 0.0f, bias = 0.0f;
#pragma unroll
        for (int i = 0; i < D / 32; ++i) {
            const int c = lane + 32 * i;
            const float x = q[h][c] * h2f_bits(ks[c]);
            const __half hi = __float2half_rn(x);
            const __half lo = __float2half_rn(x - __half2float(hi));
            qf[2 * h][c] = __half_as_ushort(hi);
            qf[2 * h + 1][c] = __half_as_ushort(lo);
            shi += __half2float(hi);
            slo += __half2float(lo);
            bias = fmaf(q[h][c], h2f_bits(kz[c]), bias);
        }
        // S = 4 (R - sum A) over both rows + sum q z (added once, on the hi row)
        cst[2 * h] = warp_sum(bias) - 4.0f * warp_sum(shi);
        cst[2 * h + 1] = -4.0f * warp_sum(slo);
    }
    __syncwarp();
    float my_cst = 0.0f;
#pragma unroll
    for (int r = 0; r < 2 * NG; ++r)
        if (g == r) my_cst = cst[r];
    uint32_t a[8][4];
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        a[s][0] = g < 2 * NG ? *reinterpret_cast<const uint32_t*>(&qf[g < 2 * NG ? g : 0][16 * s + 2 * t]) : 0u;
        a[s][2] = g < 2 * NG ? *reinterpret_cast<const uint32_t*>(&qf[g < 2 * NG ? g : 0][16 * s + 2 * t + 8]) : 0u;
        a[s][1] = a[s][3] = 0u;
    }
    __syncwarp();
    float R[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) R[n][i] = 0.0f;
    // token 8 n + g of the warp sits in word row (tl + 8 n) / 16 at code 8 (n & 1) + g
    const int qb = g >> 2, sh = 2 * (g & 3);
    const uint32_t sel = (uint32_t)qb | ((uint32_t)(2 + qb) << 4) | ((uint32_t)(4 + qb) << 8) |
                         ((uint32_t)(6 + qb) << 12);
#pragma unroll
    for (int rr = 0; rr < NT / 2; ++rr) {
        const uint32_t* row = v.kc + (size_t)(tl / 16 + rr) * D;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const uint2 w0 = *reinterpret_cast<const uint2*>(row + 16 * s + 2 * t);
            const uint2 w1 = *reinterpret_cast<const uint2*>(row + 16 * s + 2 * t + 8);
            const uint32_t y0 = __byte_perm(w0.x, w0.y, sel), y1 = __byte_perm(w1.x, w1.y, sel);
            // n = 2 rr (codes 0..7 of the row) and n = 2 rr + 1 (codes 8..15)
            const uint32_t e0 = ((y0 << (8 - sh)) & 0x03000300u) | 0x3C003C00u;
            const uint32_t e1 = ((y1 << (8 - sh)) & 0x03000300u) | 0x3C003C00u;
            const uint32_t o0 = ((y0 >> sh) & 0x03000300u) | 0x3C003C00u;
            const uint32_t o1 = ((y1 >> sh) & 0x03000300u) | 0x3C003C00u;
            mma16816(R[2 * rr], a[s], e0, e1);
            mma16816(R[2 * rr + 1], a[s], o0, o1);
        }
    }
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) S[n][jj] = fmaf(4.0f, R[n][jj], my_cst);
}

// Online softmax of the warp's logits (hi and lo rows summed first), the
// logits written out when asked; S holds p afterwards.
template <int NG, int NT>
__device__ __forceinline__ void mma_softmax(float (&S)[NT][4], int nt, MmaAcc<NG>& acc, float* lg_out,
                                            int slots) {
    constexpr int RI = MmaAcc<NG>::RI, GR = 4;
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    // hi + lo rows: lanes g = 2h and 2h + 1 both end with head h's logits
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int i = 0; i < 2 * RI; ++i) S[n][i] += __shfl_xor_sync(0xffffffffu, S[n][i], 4);
    // ---- online softmax per row; the running max moves only when it rises by
    // more than 2^8 (exact: the final division uses the same reference)
#pragma unroll
    for (int ri = 0; ri < RI; ++ri) {
        const int h = (g + 8 * ri) >> 1;
        float mx = kNegInf;
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int jj = 0; jj < 2; ++jj)
                if (8 * n + 2 * t + jj < nt) mx = fmaxf(mx, S[n][2 * ri + jj]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        float corr = 1.0f;
        if (h < NG && (acc.m[ri] == kNegInf ? mx != kNegInf : mx > acc.m[ri] + 8.0f)) {
            corr = acc.m[ri] == kNegInf ? 0.0f : ex2_approx(acc.m[ri] - mx);
            acc.m[ri] = mx;
            acc.l[ri] *= corr;
#pragma unroll
            for (int grp = 0; grp < GR; ++grp) acc.zs[ri][grp] *= corr;
        }
        // the output of head 4 ri + t sits in this lane's column: its factor comes
        // from row 2t of the block (lane 8t)
        if (__any_sync(0xffffffffu, corr != 1.0f)) {
            const float cc = __shfl_sync(0xffffffffu, corr, 8 * t);
#pragma unroll
            for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc.o[mt][ri][i] *= cc;
        }
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
                const int k = 8 * n + 2 * t + jj;
                const bool valid = h < NG && k < nt;
                if (lg_out && valid && !(g & 1)) lg_out[(size_t)h * slots + k] = S[n][2 * ri + jj];
                const float p = valid ? ex2_approx(S[n][2 * ri + jj] - acc.m[ri]) : 0.0f;
                acc.l[ri] += p;
                S[n][2 * ri + jj] = p;
            }
    }
}

// P.V of the warp's tokens over k-steps of 16, values per token (VB bits):
// D = V^T P with the value codes (times their fp16 scale) as the A operand,
// 16 channels by 16 tokens, and the probabilities (hi / lo rows) as B,
// straight from the logit accumulators.
template <int VB, int NG, int NT>
__device__ __forceinline__ void mma_pv(const View& v, int tl, int nt, const float (&S)[NT][4], MmaAcc<NG>& acc) {
    constexpr int D = 128, GR = 4;
    constexpr int RI = MmaAcc<NG>::RI;
    constexpr int vw = D * VB / 32;                      // words per token row
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const bool lo_row = (g & 1) != 0;
#pragma unroll
    for (int ks = 0; ks < NT / 2; ++ks) {
        // B: p of rows g (+ 8 ri) for tokens 2t, 2t+1 (b0) and 2t+8, 2t+9 (b1)
        uint32_t pb[RI][2];
#pragma unroll
        for (int ri = 0; ri < RI; ++ri)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const float p0 = S[2 * ks + half][2 * ri], p1 = S[2 * ks + half][2 * ri + 1];
                uint32_t x = pack_h2(p0, p1);
                if (lo_row) x = pack_h2(p0 - h2lo(x), p1 - h2hi(x));
                pb[ri][half] = x;
            }
        const int ta = tl + 16 * ks + 2 * t;
        const uint32_t* ra = v.vc + (size_t)ta * vw;
        const uint32_t* rb = ra + vw;
        const uint32_t* rc = ra + 8 * vw;
        const uint32_t* rd = rc + vw;
        // value scales of the token pairs (ta, ta+1) and (ta+8, ta+9) as f16x2 x 2^VB;
        // tokens from nt on (stale slots of the staged chunk) get scale and zero 0:
        // their p is 0 and their value must be an exact, finite 0
        uint32_t sc0[GR], sc1[GR];
        const int k0 = 16 * ks + 2 * t;
        const bool va = k0 < nt, vb = k0 + 1 < nt, vc = k0 + 8 < nt, vd = k0 + 9 < nt;
        {
            const uint2 z2 = make_uint2(0u, 0u);
            const uint2 sa = va ? *reinterpret_cast<const uint2*>(v.vs + ta * GR) : z2;
            const uint2 sb = vb ? *reinterpret_cast<const uint2*>(v.vs + (ta + 1) * GR) : z2;
            const uint2 scc = vc ? *reinterpret_cast<const uint2*>(v.vs + (ta + 8) * GR) : z2;
            const uint2 sd = vd ? *reinterpret_cast<const uint2*>(v.vs + (ta + 9) * GR) : z2;
            const __half2 mul = __float2half2_rn((float)(1 << VB));
#pragma unroll
            for (int grp = 0; grp < GR; ++grp) {
                const uint32_t wa = grp < 2 ? sa.x : sa.y, wb = grp < 2 ? sb.x : sb.y;
                const uint32_t wc = grp < 2 ? scc.x : scc.y, wd = grp < 2 ? sd.x : sd.y;
                const uint32_t sel = (grp & 1) ? 0x7632u : 0x5410u;
                const uint32_t p0 = __byte_perm(wa, wb, sel), p1 = __byte_perm(wc, wd, sel);
                const __half2 h0 = __hmul2(*reinterpret_cast<const __half2*>(&p0), mul);
                const __half2 h1 = __hmul2(*reinterpret_cast<const __half2*>(&p1), mul);
                sc0[grp] = *reinterpret_cast<const uint32_t*>(&h0);
                sc1[grp] = *reinterpret_cast<const uint32_t*>(&h1);
            }
        }
        // zero points: sum of p * z per group (hi rows carry the full p); each token's
        // four zero points in one 8-byte load
        {
            const uint2 z2 = make_uint2(0u, 0u);
            const uint2 za = va ? *reinterpret_cast<const uint2*>(v.vz + ta * GR) : z2;
            const uint2 zb = vb ? *reinterpret_cast<const uint2*>(v.vz + (ta + 1) * GR) : z2;
            const uint2 zc = vc ? *reinterpret_cast<const uint2*>(v.vz + (ta + 8) * GR) : z2;
            const uint2 zd = vd ? *reinterpret_cast<const uint2*>(v.vz + (ta + 9) * GR) : z2;
            auto zf = [](const uint2& w, int grp) -> float {
                const uint32_t x = grp < 2 ? w.x : w.y;
                return (grp & 1) ? h2hi(x) : h2lo(x);
            };
#pragma unroll
            for (int ri = 0; ri < RI; ++ri)
#pragma unroll
                for (int grp = 0; grp < GR; ++grp) {
                    const float pa0 = S[2 * ks][2 * ri], pa1 = S[2 * ks][2 * ri + 1];
                    const float pc0 = S[2 * ks + 1][2 * ri], pc1 = S[2 * ks + 1][2 * ri + 1];
                    float z = acc.zs[ri][grp];
                    z = fmaf(pa0, zf(za, grp), z);
                    z = fmaf(pa1, zf(zb, grp), z);
                    z = fmaf(pc0, zf(zc, grp), z);
                    z = fmaf(pc1, zf(zd, grp), z);
                    acc.zs[ri][grp] = z;
                }
        }
        // codes of channel c for the token pairs: f16x2 (1 + c_a / 2^VB, 1 + c_b / 2^VB)
        auto pair = [&](uint32_t wa, uint32_t wb, bool high) -> uint32_t {
            if (VB == 8) {                               // channel byte g mod 4 of the word
                const uint32_t b = (uint32_t)(g & 3);
                const uint32_t x = __byte_perm(wa, wb, b | ((4u + b) << 8)) << 2;
                return (x & 0x03FC03FCu) | 0x3C003C00u;
            } else if (VB == 4) {                        // channel nibble g of the word
                const uint32_t sel = (uint32_t)(g >> 1) | ((uint32_t)(4 + (g >> 1)) << 8);
                const uint32_t x = __byte_perm(wa, wb, sel) << (6 - 4 * (g & 1));
                return (x & 0x03C003C0u) | 0x3C003C00u;
            } else {                                     // codes g (low) and g + 8 (high) of the word
                const int q = g >> 2, sh = 2 * (g & 3);
                const uint32_t sel = (uint32_t)q | ((uint32_t)(2 + q) << 4) | ((uint32_t)(4 + q) << 8) |
                                     ((uint32_t)(6 + q) << 12);
                const uint32_t y = __byte_perm(wa, wb, sel);
                const uint32_t x = high ? (y >> sh) : (y << (8 - sh));
                return (x & 0x03000300u) | 0x3C003C00u;
            }
        };
        // s * c = 2^VB s (1 + c / 2^VB) - 2^VB s, one rounding
        auto scaled = [&](uint32_t x, uint32_t sc) -> uint32_t {
            const __half2 s2 = *reinterpret_cast<const __half2*>(&sc);
            const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&x), s2, __hneg2(s2));
            return *reinterpret_cast<const uint32_t*>(&r);
        };
        // m-tile mt: channels 16 mt + g (rows g) and 16 mt + g + 8 (rows g + 8).  The code
        // words come in 8-byte loads: words 2 mt, 2 mt + 1 (VB = 4: the low and high
        // channels of the m-tile), or words mt, mt + 1 read once for two m-tiles (VB = 2)
        uint2 xa = make_uint2(0u, 0u), xb = xa, xc = xa, xd = xa;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const int grp = mt >> 1;
            if (VB == 8) {
                // words 4 mt .. 4 mt + 3 hold the tile's 16 channels, four per word: rows g take
                // word 4 mt + g / 4, rows g + 8 word 4 mt + 2 + g / 4
                const int wo = 4 * mt + (g >> 2);
                xa = make_uint2(ra[wo], ra[wo + 2]);
                xb = make_uint2(rb[wo], rb[wo + 2]);
                xc = make_uint2(rc[wo], rc[wo + 2]);
                xd = make_uint2(rd[wo], rd[wo + 2]);
            } else if (VB == 4 || (mt & 1) == 0) {
                const int w0 = VB == 4 ? 2 * mt : mt;
                xa = *reinterpret_cast<const uint2*>(ra + w0);
                xb = *reinterpret_cast<const uint2*>(rb + w0);
                xc = *reinterpret_cast<const uint2*>(rc + w0);
                xd = *reinterpret_cast<const uint2*>(rd + w0);
            }
            auto lo = [&](const uint2& x) { return VB >= 4 ? x.x : ((mt & 1) ? x.y : x.x); };
            auto hi = [&](const uint2& x) { return VB >= 4 ? x.y : ((mt & 1) ? x.y : x.x); };
            uint32_t af[4];
            af[0] = scaled(pair(lo(xa), lo(xb), false), sc0[grp]);
            af[1] = scaled(pair(hi(xa), hi(xb), true), sc0[grp]);
            af[2] = scaled(pair(lo(xc), lo(xd), false), sc1[grp]);
            af[3] = scaled(pair(hi(xc), hi(xd), true), sc1[grp]);
#pragma unroll
            for (int ri = 0; ri < RI; ++ri) mma16816(acc.o[mt][ri], af, pb[ri][0], pb[ri][1]);
        }
    }
}

// Quad sums of l and the zero points (logit layout); then each lane takes its
// column's head (4 ri + t): hi + lo rows of o, that head's m, l and zero sums
// from lane 8t, and merges into the warp's shared-memory state.
template <int NG, int D>
__device__ __forceinline__ void flush_mma(MmaAcc<NG>& acc, Smem<NG, D>& sm) {
    constexpr int RI = MmaAcc<NG>::RI;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int ri = 0; ri < RI; ++ri) {
        acc.l[ri] += __shfl_xor_sync(0xffffffffu, acc.l[ri], 1);
        acc.l[ri] += __shfl_xor_sync(0xffffffffu, acc.l[ri], 2);
#pragma unroll
        for (int grp = 0; grp < 4; ++grp) {
            acc.zs[ri][grp] += __shfl_xor_sync(0xffffffffu, acc.zs[ri][grp], 1);
            acc.zs[ri][grp] += __shfl_xor_sync(0xffffffffu, acc.zs[ri][grp], 2);
        }
    }
#pragma unroll
    for (int ri = 0; ri < RI; ++ri) {
        const int h = 4 * ri + t;
        const float m = __shfl_sync(0xffffffffu, acc.m[ri], 8 * t);
        const float l = __shfl_sync(0xffffffffu, acc.l[ri], 8 * t);
        float zs[4];
#pragma unroll
        for (int grp = 0; grp < 4; ++grp) zs[grp] = __shfl_sync(0xffffffffu, acc.zs[ri][grp], 8 * t);
        float fo = 0.0f, fn = 0.0f, M = kNegInf, L = 0.0f;
        if (h < NG) {
            const float mo = sm.wm[warp][h];
            M = fmaxf(mo, m);
            fo = mo == kNegInf ? 0.0f : ex2_approx(mo - M);
            fn = m == kNegInf ? 0.0f : ex2_approx(m - M);
            L = sm.wl[warp][h] * fo + l * fn;
        }
        __syncwarp();                                // every lane has read the old state
        if (h < NG) {
            if (g == 0) {
                sm.wm[warp][h] = M;
                sm.wl[warp][h] = L;
            }
#pragma unroll
            for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                for (int hl = 0; hl < 2; ++hl) {
                    const int c = 16 * mt + g + 8 * hl;
                    float* p = &sm.wo[warp][h][c];
                    *p = *p * fo + (acc.o[mt][ri][2 * hl] + acc.o[mt][ri][2 * hl + 1] + zs[mt >> 1]) * fn;
                }
        }
        __syncwarp();
    }
}

// The warp's rows of query x key scales (per-channel keys), in the dynamic
// shared memory the launch reserves for them when the cache has such a tier.
template <int NG>
__device__ __forceinline__ uint16_t (&qf_rows(const DecodeArgs& a, Smem<NG, 128>& sm, int warp))[2 * NG][128] {
    uint8_t* base = reinterpret_cast<uint8_t*>(&sm) + a.qf_off + (size_t)warp * (2 * NG * 128 * sizeof(uint16_t));
    return *reinterpret_cast<uint16_t (*)[2 * NG][128]>(base);
}

// Local items [i0, i1) of a tier on the tensor cores.
template <int KB, int KAX, int VB, int NG>
__device__ void run_tier_mma(const DecodeArgs& a, Smem<NG, 128>& sm, int t, size_t unit, int r, int i0,
                             int i1, int n_local, uint8_t* stage_base, float* lg_unit, bool& ok) {
    constexpr int TPW = Cfg<NG>::TPW;
    static_assert(TPW == 16 || TPW == 32, "whole n-tile pairs per warp");
    const TierArgs& ta = a.tier[t];
    const UnitState& us = sm.us;
    const int warp = threadIdx.x >> 5;
    float qs[4][2];
    if constexpr (KAX == KVQ_AXIS_TOKEN) {
        __syncthreads();                                 // every warp is done with the previous fragments
        build_qa<KB, NG, 128>(sm, qs);
        __syncthreads();
    }
    MmaAcc<NG> acc;
#pragma unroll
    for (int ri = 0; ri < MmaAcc<NG>::RI; ++ri) {
        acc.m[ri] = kNegInf;
        acc.l[ri] = 0.0f;
#pragma unroll
        for (int grp = 0; grp < 4; ++grp) acc.zs[ri][grp] = 0.0f;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int ri = 0; ri < MmaAcc<NG>::RI; ++ri)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc.o[mt][ri][i] = 0.0f;
    for (int i = i0; i < i1; ++i) {
        ok = wait_item(a, sm, i, ok);
        if (ok) {
            const int j0 = (r + i * a.cluster - us.base[t]) * kSub;
            const int n = min(kSub, us.cnt[t] - j0);
            // per-token formats (G = 32) fold to constants; per-channel keys allow G = 32..128
            const View v = KAX == KVQ_AXIS_TOKEN
                               ? tier_view_c<KB, KVQ_AXIS_TOKEN, VB>((n + 31) & ~31, item_buf(a, stage_base, i))
                               : tier_view(ta, (n + 31) & ~31, 128, a.G, item_buf(a, stage_base, i));
            const int tl = warp * TPW;
            if (tl < n) {
                float* lo = (a.policy == KVQ_POLICY_MIKV && lg_unit) ? lg_unit + ta.slot_base + j0 + tl : nullptr;
                constexpr int NT = TPW / 8;
                float S[NT][4];
                if constexpr (KAX == KVQ_AXIS_CHANNEL)
                    mma_logits_channel<NG, NT>(v, tl, a.G, sm.q, qf_rows<NG>(a, sm, warp), S);
                else
                    mma_logits_token<KB, NG, NT>(v, tl, sm.qa, qs, S);
                const int nt = min(TPW, n - tl);
                mma_softmax<NG, NT>(S, nt, acc, lo, a.slots);
                mma_pv<VB, NG, NT>(v, tl, nt, S, acc);
            }
        }
        release_item(a, sm, unit, r, i, n_local, stage_base);
    }
    flush_mma<NG, 128>(acc, sm);
}

// ---- MiniKV format with one query head per KV head (per-channel INT2 keys,
// one scale row per 32 tokens; per-token INT2 values; D = 128, G = 32)
//
// A 2-bit code at bits 2i, 2i + 1 of a 16-bit half whose other bits are zero
// is the fp16 subnormal c * 4^i * 2^-24, exactly.  One AND with a mask thus
// turns two codes (one per half of a register) into an MMA operand, with no
// shift and no conversion; the factor 4^i * 2^-24 is shared by a whole row of
// the MMA and is taken out afterwards (keys: per token, in the logit
// epilogue; values: per channel, once at the end).  Products of fp16 numbers
// are exact in the float32 accumulators, subnormal or not.
//
// Keys: S = K Q' with the warp's 32 tokens as the M rows (two MMAs of 16
// rows), the channels in eight k-steps of 16, and Q' = q * (channel scale)
// split into fp16 hi / lo columns (N = 8: columns 0 and 1, the rest zero).
// Lane (g, t) takes byte g & 3 of the words of word row g >> 2 (tokens
// 4g .. 4g + 3 of the warp, at bits 2i of that byte) for channel pairs; one
// byte permute per pair of channels and four masks give the four tokens:
// rows g / g + 8 of MMA 0 are tokens 4g / 4g + 1, of MMA 1 tokens 4g + 2 /
// 4g + 3.  Lane (g, 0) ends with the logits of tokens 4g .. 4g + 3.
// Values: O^T = V^T P' with channels as M rows (eight M tiles), the 16
// tokens of a k-step as K, and P' = p * (the token's scale of each
// 32-channel group) as four fp16 columns, one per group.  Tile (w', P) holds
// in row g channel 16 (w' + 4 (g >> 2)) + 4 (g & 3) + 2P and in row g + 8 the
// next channel; lane (g, g >> 2) ends with both rows, in the column of their
// group.  The zero points add sum_j p_j z_j per group.

constexpr uint32_t kM0 = 0x00030003u, kM1 = 0x000C000Cu, kM2 = 0x00300030u, kM3 = 0x00C000C0u;

template <int GK>
struct Mk1Acc {
    float m, l;              // running reference max (warp-uniform), this lane's share of the sum
    float o[4][2][4];        // P.V accumulators: [word quarter w'][row pair P][fragment]
    float zs[128 / GK];      // sum of p * zero of this lane's tokens, per value group
};

template <int GK>
__device__ __forceinline__ void mk1_acc_init(Mk1Acc<GK>& acc) {
    acc.m = kNegInf;
    acc.l = 0.0f;
#pragma unroll
    for (int x = 0; x < 128 / GK; ++x) acc.zs[x] = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int P = 0; P < 2; ++P)
#pragma unroll
            for (int f = 0; f < 4; ++f) acc.o[i][P][f] = 0.0f;
}

// The staged chunk of the MiniKV format with group GK (compile-time sizes).
template <int GK>
__device__ __forceinline__ View mk1_view(int npad, const uint8_t* buf) {
    return view_of(tier_stage_sizes(KVQ_AXIS_CHANNEL, 2, 2, npad, 128, GK), buf);
}

// GK = 32 (the configs) or 16 (the MiniKV review's default): with 16, a warp's 32 tokens
// hold two key scale rows (q * scale columns 0, 1 and 2, 3 of the key MMAs, the logits of
// tokens 16..31 in lanes t = 1) and the values eight 16-channel groups (all eight B
// columns of the P.V MMAs).
// Shared-memory strides chosen so that the lanes of one fragment load hit distinct banks: a
// query piece (hi or lo of one key scale row: [k-step][t][reg], 64 words) every 72 words, a
// value group's 32 fp16 (p x scale) every 40 halves.
constexpr int kQfPiece = 72, kPsGroup = 40;

template <int GK>
struct Mk1Ctx {
    uint32_t* qf;            // this warp's query fragments, one piece every kQfPiece words
    float* pw;               // this warp's 32 probabilities
    uint16_t* psw;           // probability x value scale, fp16, one group every kPsGroup halves
    const uint2* qfb;        // B-fragment source of the key MMAs (a query piece)
    const uint32_t* psb;     // B-fragment source of the P.V MMAs (a value group)
    float4 q4;               // query channels 4 lane .. 4 lane + 3 (base-2 scaled)
    uint32_t bsel;           // byte permute of lane group g (key codes)
    uint32_t vsel;           // byte permute of the value codes (operands swapped for t >= 2)
    int voff;                // word offset of the first value row a lane loads (t >= 2: the second)
    int tv;                  // the lane t that holds lane group g's logits
};

// Bytes of a warp's query fragments and (groups of 16) value-group products.
template <int GK>
constexpr uint32_t mk1_qf_warp_bytes() {
    return GK == 32 ? 2u * kQfPiece * 4u : 4u * kQfPiece * 4u + 8u * kPsGroup * 2u;
}

template <int GK>
__device__ __forceinline__ Mk1Ctx<GK> mk1_ctx(const DecodeArgs& a, Smem<1, 128>& sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    constexpr int NKR = 32 / GK, NGV = 128 / GK;
    Mk1Ctx<GK> x;
    // probabilities (32 floats) and probability x value scale: over the probabilities for
    // GK = 32, after the fragments for GK = 16
    x.qf = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(&sm) + a.qf_off +
                                       (size_t)warp * mk1_qf_warp_bytes<GK>());
    x.pw = &sm.lg[warp][0][0];
    x.psw = GK == 32 ? reinterpret_cast<uint16_t*>(x.pw) : reinterpret_cast<uint16_t*>(x.qf + 4 * kQfPiece);
    // column g of the B fragments: the query piece / value group g; columns past them feed
    // MMA outputs nobody reads, so those lanes repeat a real piece / group (finite values,
    // and their loads coincide with another lane's)
    x.qfb = reinterpret_cast<const uint2*>(x.qf + (g & (2 * NKR - 1)) * kQfPiece) + t;
    x.psb = reinterpret_cast<const uint32_t*>(x.psw + (g & (NGV - 1)) * kPsGroup) + t;
    x.tv = GK == 32 ? 0 : (g >> 2);
    x.q4 = *reinterpret_cast<const float4*>(&sm.q[0][4 * lane]);
    x.bsel = (uint32_t)(g & 3) | ((uint32_t)(4 + (g & 3)) << 8);
    x.vsel = t >= 2 ? ((uint32_t)(4 + (g & 3)) | ((uint32_t)(g & 3) << 8)) : x.bsel;
    x.voff = t >= 2 ? 8 : 0;
    return x;
}

// This warp's tokens [tl, tl + nt) (nt <= 32) of a staged chunk: logits, online softmax
// and P.V into acc.
template <int GK>
__device__ __forceinline__ void mk1_item(const View& v, int tl, int nt, const Mk1Ctx<GK>& x, Mk1Acc<GK>& acc) {
    constexpr int NKR = 32 / GK, NGV = 128 / GK;
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const float4 q4 = x.q4;
    // -- Q' = q * scale of each key scale row, as hi / lo fp16 fragments, and sum_c q z
    float bias[NKR];
#pragma unroll
    for (int kr = 0; kr < NKR; ++kr) {
        const size_t ro = (size_t)(tl / GK + kr) * 128 + 4 * lane;
        const uint2 s2 = *reinterpret_cast<const uint2*>(v.ks + ro);
        const uint2 z2 = *reinterpret_cast<const uint2*>(v.kz + ro);
        const float x0 = q4.x * h2lo(s2.x), x1 = q4.y * h2hi(s2.x);
        const float x2 = q4.z * h2lo(s2.y), x3 = q4.w * h2hi(s2.y);
        const uint32_t hi01 = pack_h2(x0, x1), hi23 = pack_h2(x2, x3);
        const uint32_t lo01 = pack_h2(x0 - h2lo(hi01), x1 - h2hi(hi01));
        const uint32_t lo23 = pack_h2(x2 - h2lo(hi23), x3 - h2hi(hi23));
        bias[kr] = fmaf(q4.x, h2lo(z2.x), fmaf(q4.y, h2hi(z2.x), fmaf(q4.z, h2lo(z2.y), q4.w * h2hi(z2.y))));
        // the MMA's k = 2t, 2t + 1, 2t + 8, 2t + 9 of k-step s are channels 16 s + 4t .. + 3:
        // lane 4s + t holds exactly the B registers of lane t at k-step s
        uint32_t* qh = x.qf + 2 * kQfPiece * kr;
        reinterpret_cast<uint2*>(qh)[lane] = make_uint2(hi01, hi23);
        reinterpret_cast<uint2*>(qh + kQfPiece)[lane] = make_uint2(lo01, lo23);
        bias[kr] = warp_sum(bias[kr]);
    }
    const float bias_g = NKR == 1 ? bias[0] : ((g >> 2) ? bias[NKR - 1] : bias[0]);
    __syncwarp();
    // -- logits: two MMAs (tokens 4g + {0, 1} and 4g + {2, 3}), each over two accumulator
    // chains of four k-steps
    float R[2][2][4];
#pragma unroll
    for (int P = 0; P < 2; ++P)
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int f = 0; f < 4; ++f) R[P][e][f] = 0.0f;
    {
        const uint32_t* rowp = v.kc + (size_t)((tl >> 4) + (g >> 2)) * 128;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            // channels 16 s + 4t .. + 3 (the k order above): one 16-byte load
            const uint4 w = *reinterpret_cast<const uint4*>(rowp + 16 * s + 4 * t);
            const uint2 b = x.qfb[s * 4];
            const uint32_t y0 = __byte_perm(w.x, w.y, x.bsel), y1 = __byte_perm(w.z, w.w, x.bsel);
            const uint32_t a0[4] = {y0 & kM0, y0 & kM1, y1 & kM0, y1 & kM1};
            const uint32_t a1[4] = {y0 & kM2, y0 & kM3, y1 & kM2, y1 & kM3};
            mma16816(R[0][s & 1], a0, b.x, b.y);
            mma16816(R[1][s & 1], a1, b.x, b.y);
        }
    }
    // -- logits of tokens 4g + j (lanes t == tv): code factor 4^j * 2^-24 out, bias in
    float lg[4];
    lg[0] = fmaf((R[0][0][0] + R[0][1][0]) + (R[0][0][1] + R[0][1][1]), 16777216.0f, bias_g);  // 2^24
    lg[1] = fmaf((R[0][0][2] + R[0][1][2]) + (R[0][0][3] + R[0][1][3]), 4194304.0f, bias_g);   // 2^22
    lg[2] = fmaf((R[1][0][0] + R[1][1][0]) + (R[1][0][1] + R[1][1][1]), 1048576.0f, bias_g);   // 2^20
    lg[3] = fmaf((R[1][0][2] + R[1][1][2]) + (R[1][0][3] + R[1][1][3]), 262144.0f, bias_g);    // 2^18
    bool valid[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) valid[j] = t == x.tv && 4 * g + j < nt;
    float mx = fmaxf(fmaxf(valid[0] ? lg[0] : kNegInf, valid[1] ? lg[1] : kNegInf),
                     fmaxf(valid[2] ? lg[2] : kNegInf, valid[3] ? lg[3] : kNegInf));
    // the reference moves only when the max rises by more than 2^8 (exact: the final
    // division uses the same reference); the warp's max is formed only then
    if (__any_sync(0xffffffffu, acc.m == kNegInf ? mx != kNegInf : mx > acc.m + 8.0f)) {
        if (GK != 32) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        mx = __shfl_sync(0xffffffffu, mx, 0);
        const float corr = acc.m == kNegInf ? 0.0f : ex2_approx(acc.m - mx);
        acc.m = mx;
        acc.l *= corr;
#pragma unroll
        for (int k = 0; k < NGV; ++k) acc.zs[k] *= corr;
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int P = 0; P < 2; ++P)
#pragma unroll
                for (int f = 0; f < 4; ++f) acc.o[k][P][f] *= corr;
    }
    {
        float4 p;
        p.x = valid[0] ? ex2_approx(lg[0] - acc.m) : 0.0f;
        p.y = valid[1] ? ex2_approx(lg[1] - acc.m) : 0.0f;
        p.z = valid[2] ? ex2_approx(lg[2] - acc.m) : 0.0f;
        p.w = valid[3] ? ex2_approx(lg[3] - acc.m) : 0.0f;
        acc.l += (p.x + p.y) + (p.z + p.w);
        if (t == x.tv) *reinterpret_cast<float4*>(x.pw + 4 * g) = p;
    }
    __syncwarp();
    // -- lane = token: p times each group's value scale into [group][token], and the zero
    // points (stale slots past nt read as zero scale and zero point)
    {
        const float p = x.pw[lane];
        __syncwarp();                                    // every lane has its p: ps may overwrite pw
        const bool ok_t = lane < nt;
        uint32_t sw[NGV / 2], zw[NGV / 2];
        if constexpr (NGV == 4) {
            const uint2 s2 = *reinterpret_cast<const uint2*>(v.vs + (size_t)(tl + lane) * 4);
            const uint2 z2 = *reinterpret_cast<const uint2*>(v.vz + (size_t)(tl + lane) * 4);
            sw[0] = s2.x; sw[1] = s2.y; zw[0] = z2.x; zw[1] = z2.y;
        } else {
            const uint4 s4 = *reinterpret_cast<const uint4*>(v.vs + (size_t)(tl + lane) * 8);
            const uint4 z4 = *reinterpret_cast<const uint4*>(v.vz + (size_t)(tl + lane) * 8);
            sw[0] = s4.x; sw[1] = s4.y; sw[2] = s4.z; sw[3] = s4.w;
            zw[0] = z4.x; zw[1] = z4.y; zw[2] = z4.z; zw[3] = z4.w;
        }
#pragma unroll
        for (int e = 0; e < NGV / 2; ++e) {
            sw[e] = ok_t ? sw[e] : 0u;
            zw[e] = ok_t ? zw[e] : 0u;
            const uint32_t ps2 = pack_h2(p * h2lo(sw[e]), p * h2hi(sw[e]));
            x.psw[(2 * e) * kPsGroup + lane] = (uint16_t)(ps2 & 0xffffu);
            x.psw[(2 * e + 1) * kPsGroup + lane] = (uint16_t)(ps2 >> 16);
            acc.zs[2 * e] = fmaf(p, h2lo(zw[e]), acc.zs[2 * e]);
            acc.zs[2 * e + 1] = fmaf(p, h2hi(zw[e]), acc.zs[2 * e + 1]);
        }
    }
    __syncwarp();
    // -- P.V over two k-steps of 16 tokens: B = (p s) of tokens 16 ks + 2t, + 1 (b0) and
    // + 8, + 9 (b1) in column g (value group g).  Lanes t >= 2 load the rows of tokens
    // k0 + 1 and k0 first (no bank shared with lanes t < 2) and swap the permute's operands.
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
        const int k0 = 16 * ks + 2 * t;
        const uint32_t b0 = x.psb[8 * ks], b1 = x.psb[8 * ks + 4];
        const uint32_t* vrow = v.vc + (size_t)(tl + k0) * 8 + 4 * (g >> 2);
        const uint4 xa = *reinterpret_cast<const uint4*>(vrow + x.voff);
        const uint4 xb = *reinterpret_cast<const uint4*>(vrow + (8 - x.voff));
        const uint4 xc = *reinterpret_cast<const uint4*>(vrow + 64 + x.voff);
        const uint4 xd = *reinterpret_cast<const uint4*>(vrow + (72 - x.voff));
        const uint32_t wa[4] = {xa.x, xa.y, xa.z, xa.w}, wb[4] = {xb.x, xb.y, xb.z, xb.w};
        const uint32_t wc[4] = {xc.x, xc.y, xc.z, xc.w}, wd[4] = {xd.x, xd.y, xd.z, xd.w};
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const uint32_t ya = __byte_perm(wa[w], wb[w], x.vsel), yc = __byte_perm(wc[w], wd[w], x.vsel);
            const uint32_t a0[4] = {ya & kM0, ya & kM1, yc & kM0, yc & kM1};
            const uint32_t a1[4] = {ya & kM2, ya & kM3, yc & kM2, yc & kM3};
            mma16816(acc.o[w][0], a0, b0, b1);
            mma16816(acc.o[w][1], a1, b0, b1);
        }
    }
    __syncwarp();                                        // pw / ps / qf are rewritten by the next item
}

// The warp's state merged into its shared-memory state (sm.wm / wl / wo of this warp).
template <int GK>
__device__ __forceinline__ void mk1_flush(Mk1Acc<GK>& acc, Smem<1, 128>& sm) {
    constexpr int NGV = 128 / GK;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    acc.l = warp_sum(acc.l);
#pragma unroll
    for (int k = 0; k < NGV; ++k) acc.zs[k] = warp_sum(acc.zs[k]);
    float fo = 0.0f, fn = 0.0f;
    {
        const float mo = sm.wm[warp][0];
        const float M = fmaxf(mo, acc.m);
        fo = mo == kNegInf ? 0.0f : ex2_approx(mo - M);
        fn = acc.m == kNegInf ? 0.0f : ex2_approx(acc.m - M);
        __syncwarp();
        if (lane == 0) {
            sm.wl[warp][0] = sm.wl[warp][0] * fo + acc.l * fn;
            sm.wm[warp][0] = M;
        }
    }
    // tile (w', P) row g holds channel 16 (w' + 4 (g >> 2)) + 4 (g & 3) + 2P, row g + 8 the
    // next; their value group n (column n of the MMA) sits in lane t = n / 2, slot n mod 2
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        constexpr int kQ = 64 / GK;                      // groups per 64 channels
        const int n0 = (16 * w) / GK;                    // the group for g < 4; g >= 4 adds kQ
        const int n = n0 + ((g >> 2) ? kQ : 0);
        if (t != (n >> 1)) continue;
        const int slot = n & 1;
        const float zg = (g >> 2) ? acc.zs[n0 + kQ] : acc.zs[n0];
#pragma unroll
        for (int P = 0; P < 2; ++P) {
            const int c = 16 * (w + 4 * (g >> 2)) + 4 * (g & 3) + 2 * P;
            const float lo_row = (P ? 1048576.0f : 16777216.0f);  // 2^(24 - 4P)
            const float o0 = fmaf(slot ? acc.o[w][P][1] : acc.o[w][P][0], lo_row, zg);
            const float o1 = fmaf(slot ? acc.o[w][P][3] : acc.o[w][P][2], 0.25f * lo_row, zg);
            float* dst = &sm.wo[warp][0][c];
            dst[0] = dst[0] * fo + o0 * fn;
            dst[1] = dst[1] * fo + o1 * fn;
        }
    }
    __syncwarp();
}

// Local items [i0, i1) of the MiniKV tier, one query head per KV head.
template <int NG, int GK>
__device__ void run_tier_mk1(const DecodeArgs& a, Smem<NG, 128>& sm, int tier, size_t unit, int r, int i0,
                             int i1, int n_local, uint8_t* stage_base, bool& ok) {
    static_assert(NG == 1, "one query head per KV head");
    static_assert(GK == 32 || GK == 16, "groups of 32 or 16");
    constexpr int TPW = Cfg<NG>::TPW;
    static_assert(TPW == 32, "32 tokens per warp and item");
    constexpr int NGV = 128 / GK;
    const UnitState& us = sm.us;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Mk1Ctx<GK> x = mk1_ctx<GK>(a, sm);
    // the copies of this tier's next items, one array per lane (lanes 0..5): a chunk of npad
    // tokens stages array k at bytes [off_k npad, off_k npad + bytes_k npad) of its buffer,
    // from base_k + (chunk index) * 128 bytes_k (compile-time sizes of the format)
    constexpr uint32_t kSB = 256 / GK;           // scale (or zero) bytes per token, keys and values
    const TierArgs& ta = a.tier[tier];
    const uint8_t* cp_src = nullptr;
    uint32_t cp_off = 0u, cp_bpt = 0u;
    {
        const size_t cap = (size_t)ta.cap;
        switch (lane) {
            case 0: cp_src = reinterpret_cast<const uint8_t*>(ta.k_codes + unit * (cap / 16) * 128); cp_off = 0; cp_bpt = 32; break;
            case 1: cp_src = reinterpret_cast<const uint8_t*>(ta.k_scale + unit * (cap / GK) * 128); cp_off = 32; cp_bpt = kSB; break;
            case 2: cp_src = reinterpret_cast<const uint8_t*>(ta.k_zero + unit * (cap / GK) * 128); cp_off = 32 + kSB; cp_bpt = kSB; break;
            case 3: cp_src = reinterpret_cast<const uint8_t*>(ta.v_codes + unit * cap * 8); cp_off = 32 + 2 * kSB; cp_bpt = 32; break;
            case 4: cp_src = reinterpret_cast<const uint8_t*>(ta.v_scale + unit * cap * NGV); cp_off = 64 + 2 * kSB; cp_bpt = kSB; break;
            case 5: cp_src = reinterpret_cast<const uint8_t*>(ta.v_zero + unit * cap * NGV); cp_off = 64 + 3 * kSB; cp_bpt = kSB; break;
            default: break;
        }
    }
    Mk1Acc<GK> acc;
    mk1_acc_init(acc);
    for (int i = i0; i < i1; ++i) {
        ok = wait_item(a, sm, i, ok);
        const int j0 = (r + i * a.cluster - us.base[tier]) * kSub;
        const int n = min(kSub, us.cnt[tier] - j0);
        const int tl = warp * TPW;
        if (ok && tl < n)
            mk1_item<GK>(mk1_view<GK>((n + 31) & ~31, item_buf(a, stage_base, i)), tl, min(TPW, n - tl), x, acc);
        // every warp is done with item i: warp 0 requests item i + S into its buffer, the six
        // copies of a chunk of this tier side by side (other items: the general path)
        __syncthreads();
        if (warp == 0 && i + a.stages < n_local && !sm.fail) {
            const int inext = i + a.stages, kn = r + inext * a.cluster;
            if (kn < us.base[tier + 1]) {
                const int idx = kn - us.base[tier];
                const int np = (min(kSub, us.cnt[tier] - idx * kSub) + 31) & ~31;
                const int sb = inext & (a.stages - 1);
                const uint32_t bar = smem_u32(&sm.bar[sb]);
                if (lane == 0) mbar_expect_tx(bar, (64u + 4u * kSB) * (uint32_t)np);
                __syncwarp();
                if (lane < 6)
                    bulk_load(smem_u32(stage_base) + (uint32_t)sb * a.stage_bytes + cp_off * (uint32_t)np,
                              cp_src + (size_t)idx * (kSub * cp_bpt), cp_bpt * (uint32_t)np, bar);
            } else if (lane == 0) {
                issue_item(a, us, unit, r, inext, stage_base, sm.bar);
            }
            if (lane == 0) sm.issued = inext + 1;
        }
    }
    mk1_flush<GK>(acc, sm);
}

// FAM selects the formats compiled into one kernel: bit 0 keys per channel
// (MiniKV), bit 1 keys per token (DiffKV, MiKV tiers).
template <int NG, int D, int FAM>
__device__ void dispatch_tier(const DecodeArgs& a, Smem<NG, D>& sm, int t, size_t unit, int r, int i0,
                              int i1, int n_local, uint8_t* stage, float* lg_unit, bool& ok) {
    const TierArgs& ta = a.tier[t];
    const int kb = ta.k_bits, vb = ta.v_bits, ax = ta.k_axis;
    if ((FAM & 1) && ax == KVQ_AXIS_CHANNEL && kb == 2 && vb == 2) {
        if constexpr (D == 128 && NG == 1) {
            if (a.G == 16) run_tier_mk1<NG, 16>(a, sm, t, unit, r, i0, i1, n_local, stage, ok);
            else run_tier_mk1<NG, 32>(a, sm, t, unit, r, i0, i1, n_local, stage, ok);
        }
        else if constexpr (D == 128 && NG <= 4)
            run_tier_mma<2, KVQ_AXIS_CHANNEL, 2, NG>(a, sm, t, unit, r, i0, i1, n_local, stage, lg_unit, ok);
        else
            run_tier<2, KVQ_AXIS_CHANNEL, 2, D, NG>(a, sm, t, unit, r, i0, i1, n_local, stage, lg_unit, ok);
        return;
    }
    if constexpr ((FAM & 2) && D == 128 && NG >= 2) {
        if (ax == KVQ_AXIS_TOKEN && kb == 8 && vb == 4) { run_tier_mma<8, KVQ_AXIS_TOKEN, 4, NG>(a, sm, t, unit, r, i0, i1, n_local, stage, lg_unit, ok); return; }
        if (ax == KVQ_AXIS_TOKEN && kb == 4 && vb == 8) { run_tier_mma<4, KVQ_AXIS_TOKEN, 8, NG>(a, sm, t, unit, r, i0, i1, n_local, stage, lg_unit, ok); return; }
        if (ax == KVQ_AXIS_TOKEN && kb == 4 && vb == 2) { run_tier_mma<4, KVQ_AXIS_TOKEN, 2, NG>(a, sm, t, unit, r, i0, i1, n_local, stage, lg_unit, ok); return; }
        if (ax == KVQ_AXIS_TOKEN && kb == 4 && vb == 4) { run_tier_mma<4, KVQ_AXIS_TOKEN, 4, NG>(a, sm, t, unit, r, i0, i1, n_local, stage, lg_unit, ok); return; }
        if (ax == KVQ_AXIS_TOKEN && kb == 2 && vb == 2) { run_tier_mma<2, KVQ_AXIS_TOKEN, 2, NG>(a, sm, t, unit, r, i0, i1, n_local, stage, lg_unit, ok); return; }
    } else if constexpr ((FAM & 2) && D == 128) {
        if (ax == KVQ_AXIS_TOKEN && kb == 8 && vb == 4) { run_tier<8, KVQ_AXIS_TOKEN, 4, D, NG>(a, sm, t, unit, r, i0, i1, n_local, stage, lg_unit, ok); return; }
        if (ax == KVQ_AXIS_TOKEN && kb == 4 && vb == 8) { run_tier<4, KVQ_AXIS_TOKEN, 8, D, NG>(a, sm, t, unit, r, i0, i1, n_local, stage, lg_unit, ok); return; }
        if (ax == KVQ_AXIS_TOKEN && kb == 4 && vb == 2) { run_tier<4, KVQ_AXIS_TOKEN, 2, D, NG>(a, sm, t, unit, r, i0, i1, n_local, stage, lg_unit, ok); return; }
        if (ax == KVQ_AXIS_TOKEN && kb == 4 && vb == 4) { run_tier<4, KVQ_AXIS_TOKEN, 4, D, NG>(a, sm, t, unit, r, i0, i1, n_local, stage, lg_unit, ok); return; }
        if (ax == KVQ_AXIS_TOKEN && kb == 2 && vb == 2) { run_tier<2, KVQ_AXIS_TOKEN, 2, D, NG>(a, sm, t, unit, r, i0, i1, n_local, stage, lg_unit, ok); return; }
    }
    // a format without a kernel (the host validation lists exactly the built ones):
    // consume the items so that the staging stays in step
    if (threadIdx.x == 0) atomicOr(&g_status_decode, kDevCheck);
    for (int i = i0; i < i1; ++i) {
        ok = wait_item(a, sm, i, ok);
        release_item(a, sm, unit, r, i, n_local, stage);
    }
}

// Local items [i0, i1) of the residual ring.
template <int NG, int D>
__device__ void run_residual(const DecodeArgs& a, Smem<NG, D>& sm, size_t unit, int r, int i0, int i1,
                             int n_local, uint8_t* stage_base, float* lg_unit, bool& ok) {
    const UnitState& us = sm.us;
    const int warp = threadIdx.x >> 5;
    const bool bf = a.bf16 != 0;
    WarpAcc<NG, D / 32> acc;
    acc_init(acc);
    for (int i = i0; i < i1; ++i) {
        ok = wait_item(a, sm, i, ok);
        if (ok) {
            const int j0 = (r + i * a.cluster - us.base[a.n_tiers]) * kResItem;
            const int n = min(kResItem, us.len + 1 - j0);
            const uint8_t* buf = item_buf(a, stage_base, i);
            const uint16_t* rk = reinterpret_cast<const uint16_t*>(buf);
            const uint16_t* rv = reinterpret_cast<const uint16_t*>(buf + a16((uint32_t)n * D * 2));
            const int w0 = warp * Cfg<NG>::RPW;
            if (w0 < n) {
                float* lo = (lg_unit && a.policy != KVQ_POLICY_MINIKV) ? lg_unit + a.res_slot_base + j0 + w0 : nullptr;
                residual_rows<NG, D>(sm, rk + (size_t)w0 * D, rv + (size_t)w0 * D, min(Cfg<NG>::RPW, n - w0), bf,
                                     acc, lo, a.slots);
            }
        }
        release_item(a, sm, unit, r, i, n_local, stage_base);
    }
    flush_lane_values<NG, D>(acc, sm);
}

// ---- policy work after the merge

// DiffKV: this step's attention added to the window scores of the CTA's own
// ring rows, every (item, row, head) at once, all loads in flight together.
template <int NG, int D>
__device__ void add_scores(const DecodeArgs& a, const Smem<NG, D>& sm, size_t unit, int r, int n_local,
                           const float* lg_unit) {
    const UnitState& us = sm.us;
    const int b = (int)(unit / a.Hkv), hkv = (int)(unit % a.Hkv);
    const int cap = a.res_cap;
    const float* lse2 = sm.lse2;
    const int i_res = local_at(us.base[a.n_tiers], r, a.cluster);   // first local ring item
    const int n_pairs = (n_local - i_res) * kResItem * NG;
    for (int x = threadIdx.x; x < n_pairs; x += blockDim.x) {
        const int k = x / (kResItem * NG), rem = x % (kResItem * NG);
        int idx;
        (void)item_kind(us, a.n_tiers, r + (i_res + k) * a.cluster, idx);
        const int li = idx * kResItem + rem / NG, h = rem % NG;
        if (li > us.len) continue;                               // past the new token
        const float p = ex2_approx(__ldcg(lg_unit + (size_t)h * a.slots + a.res_slot_base + li) - lse2[h]);
        float* wa = a.win_acc + ((size_t)b * a.Hq + hkv * NG + h) * cap + (us.start + li) % cap;
        *wa = li < us.len ? __fadd_rn(*wa, p) : p;
    }
}

// MiKV: this step's attention added to the cumulative score of every token,
// once the step's lse is known (written by the decode launch with the ring
// state it saw).  One thread per logits slot of a unit: the tiers' slots,
// then the ring's; p = sum over the group's heads of 2^(s - lse2).
struct ScoreArgs {
    int g, n_tiers, slots, res_cap, res_slot_base, score_cap;
    const int32_t* token_id[KVQ_MAX_TIERS];
    const int32_t* count[KVQ_MAX_TIERS];
    int cap[KVQ_MAX_TIERS], slot_base[KVQ_MAX_TIERS];
    const int32_t* res_token_id;
    const float* logits;
    const float* lse2;
    const int32_t* meta;
    float* cum_score;
};

__global__ void __launch_bounds__(256) mikv_scores_kernel(ScoreArgs s) {
    const size_t unit = blockIdx.y;
    const int x = (int)(blockIdx.x * blockDim.x + threadIdx.x);
    if (x >= s.slots) return;
    const int32_t* meta = s.meta + unit * 4;
    int id;
    bool fresh = false;
    if (x >= s.res_slot_base) {
        const int li = x - s.res_slot_base, len = meta[0];
        if (li > len) return;
        id = li < len ? s.res_token_id[unit * (size_t)s.res_cap + (meta[1] + li) % s.res_cap] : meta[2];
        fresh = li == len;                     // the step's own token: its first score
    } else {
        static_assert(KVQ_MAX_TIERS == 2, "two tiers at most");
        const bool t1 = s.n_tiers > 1 && x >= s.slot_base[1];     // no indexing of the parameter arrays
        const int cap = t1 ? s.cap[1] : s.cap[0];
        const int j = x - (t1 ? s.slot_base[1] : s.slot_base[0]);
        const int n = min(max((t1 ? s.count[1] : s.count[0])[unit], 0), cap);
        if (j >= n) return;
        id = (t1 ? s.token_id[1] : s.token_id[0])[unit * (size_t)cap + j];
    }
    const float* lg = s.logits + unit * (size_t)s.g * s.slots + x;
    float p = 0.0f;
    for (int h = 0; h < s.g; ++h) p += ex2_approx(__ldcs(lg + (size_t)h * s.slots) - s.lse2[unit * 8 + h]);
    if (id < 0 || id >= s.score_cap) {
        atomicOr(&g_status_decode, kDevCheck);
        return;
    }
    float* cs = s.cum_score + unit * (size_t)s.score_cap + id;
    *cs = fresh ? p : __fadd_rn(*cs, p);
}

// Leader, MiniKV: the G oldest residual tokens (the new one already in the
// ring) move to tier 0 -- keys grouped per channel along tokens, values per
// token along channels.  Returns false when tier 0 is full.
template <typename T>
__device__ bool minikv_flush(const DecodeArgs& a, size_t unit, int start, int cnt) {
    const TierArgs& t = a.tier[0];
    const int G = a.G, D = a.D, cap = a.res_cap;
    if (cnt + G > t.cap) return false;
    const T* rk = reinterpret_cast<const T*>(a.res_k);
    const T* rv = reinterpret_cast<const T*>(a.res_v);
    const size_t rb = unit * (size_t)cap;
    auto row = [&](int i) { return rk + (rb + (start + i) % cap) * D; };
    uint32_t* codes = t.k_codes + (unit * (size_t)(t.cap * t.k_bits / 32) + cnt * t.k_bits / 32) * D;
    uint16_t* s = t.k_scale + (unit * (size_t)(t.cap / G) + cnt / G) * D;
    uint16_t* z = t.k_zero + (unit * (size_t)(t.cap / G) + cnt / G) * D;
    for (int c = threadIdx.x; c < D; c += blockDim.x)
        quant_channel_group<T>(row, G, c, t.k_bits, codes, D, s + c, z + c);
    const int groups = D / G;
    for (int x = threadIdx.x; x < G * groups; x += blockDim.x) {
        const int i = x / groups, grp = x % groups;
        const T* src = rv + (rb + (start + i) % cap) * D + (size_t)grp * G;
        const size_t slot = unit * (size_t)t.cap + cnt + i;
        quant_token_group([&](int k) { return Elem<T>::to_f(src[k]); }, G, t.v_bits,
                          t.v_codes + slot * (D * t.v_bits / 32) + grp * (G * t.v_bits / 32),
                          t.v_scale + slot * groups + grp, t.v_zero + slot * groups + grp);
    }
    for (int i = threadIdx.x; i < G; i += blockDim.x)
        t.token_id[unit * (size_t)t.cap + cnt + i] = a.res_token_id[rb + (start + i) % cap];
    return true;
}

// ---- the kernel

// Grid = (C, units), cluster (C, 1, 1): CTA r of the cluster of unit u.
template <int NG, int D, int FAM>
__global__ void __launch_bounds__(Cfg<NG>::kThreads, Cfg<NG>::MINB) decode_kernel(DecodeArgs a) {
    constexpr int W = Cfg<NG>::W;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem<NG, D>& sm = *reinterpret_cast<Smem<NG, D>*>(smem_raw);
    float* part = reinterpret_cast<float*>(smem_raw + a.part_off);   // leader: [C][NG][D + 2]
    uint8_t* stage_base = smem_raw + a.stage_off;
    const int C = a.cluster;
    const int r = blockIdx.x;
    const int ir = C - 1 - r;                   // item rank: the leader, which also merges, takes the last share
    const size_t unit = blockIdx.y;
    const int b = (int)(unit / a.Hkv), hkv = (int)(unit % a.Hkv);
    const bool bf = a.bf16 != 0;

    cluster_arrive_relaxed();                   // "started": the leader's shared memory exists
    if (threadIdx.x == 32) prefetch_start(a, unit, ir);
    if (threadIdx.x == 0) {
        UnitState& us = sm.us;
        // all counters requested at once, then checked
        int raw[KVQ_MAX_TIERS];
#pragma unroll
        for (int t = 0; t < KVQ_MAX_TIERS; ++t) raw[t] = t < a.n_tiers ? a.tier[t].count[unit] : 0;
        const int rl = a.res_len[unit], rs = a.res_start[unit], ps = a.pos[unit];
        bool bad = false;
        us.base[0] = 0;
#pragma unroll
        for (int t = 0; t < KVQ_MAX_TIERS; ++t) {
            if (t >= a.n_tiers) break;
            const int n = min(max(raw[t], 0), a.tier[t].cap);
            bad |= raw[t] != n;
            us.cnt[t] = n;
            us.base[t + 1] = us.base[t] + (n + kSub - 1) / kSub;
        }
        const int cap = a.res_cap;
        us.len = min(max(rl, 0), cap - 1);
        us.start = min(max(rs, 0), cap - 1);
        bad |= rl != us.len || rs != us.start;
        us.pos = ps;
        us.total = us.base[a.n_tiers] + (us.len + 1 + kResItem - 1) / kResItem;
        if (bad) atomicOr(&g_status_decode, kDevCheck);
        for (int st = 0; st < a.stages; ++st) mbar_init(smem_u32(&sm.bar[st]), 1);
        sm.fail = 0;
        fence_mbar_init();
        const int n_local = us.total > ir ? (us.total - ir + C - 1) / C : 0;
        for (int i = 0; i < a.stages && i < n_local; ++i)
            if (!(i == 0 && ir == 0 && (int)unit == a.withhold_unit)) issue_item(a, us, unit, ir, i, stage_base, sm.bar);
        sm.issued = min(a.stages, n_local);
    }
    for (int x = threadIdx.x; x < NG * D; x += blockDim.x) {
        const int h = x / D, c = x % D;
        sm.q[h][c] = ldf(a.q, ((size_t)b * a.Hq + (size_t)hkv * NG + h) * D + c, bf) * a.scale_log2;
    }
    for (int x = threadIdx.x; x < W * NG; x += blockDim.x) {
        sm.wm[x / NG][x % NG] = kNegInf;
        sm.wl[x / NG][x % NG] = 0.0f;
    }
    for (int x = threadIdx.x; x < W * NG * D; x += blockDim.x) (&sm.wo[0][0][0])[x] = 0.0f;
    __syncthreads();

    const UnitState& us = sm.us;
    // the new token joins the ring now, off the leader's final path: its slot
    // (start + len) is not among the len rows any CTA reads this step (the new
    // row itself is read from k_new / v_new), and the leader's MiniKV flush
    // reads it after the cluster barriers of the merge
    if (r == C - 1) {
        const int cap = a.res_cap;
        const size_t slot = unit * (size_t)cap + (us.start + us.len) % cap;
        for (int c = threadIdx.x; c < D; c += blockDim.x) {
            stf(a.res_k, slot * D + c, ldf(a.k_new, unit * D + c, bf), bf);
            stf(a.res_v, slot * D + c, ldf(a.v_new, unit * D + c, bf), bf);
        }
        if (threadIdx.x == 0) a.res_token_id[slot] = us.pos;
    }
    const int n_local = us.total > ir ? (us.total - ir + C - 1) / C : 0;
    float* lg_unit = a.logits ? a.logits + unit * NG * (size_t)a.slots : nullptr;
    bool ok = true;
    for (int t = 0; t < a.n_tiers; ++t) {
        const int i0 = local_at(us.base[t], ir, C), i1 = local_at(us.base[t + 1], ir, C);
        if (i1 > i0) dispatch_tier<NG, D, FAM>(a, sm, t, unit, ir, i0, i1, n_local, stage_base, lg_unit, ok);
    }
    {
        const int i0 = local_at(us.base[a.n_tiers], ir, C);
        if (n_local > i0) run_residual<NG, D>(a, sm, unit, ir, i0, n_local, n_local, stage_base, lg_unit, ok);
    }
    __syncthreads();
    if (sm.fail && threadIdx.x == 0) {
        atomicOr(&g_status_decode, kDevTimeout);
        // let every copy still in flight land before the buffers go away: the last
        // item requested into each buffer (items are requested in order)
        const int S = a.stages, n = sm.issued;
        for (int i = max(0, n - S); i < n; ++i)
            (void)mbar_wait(smem_u32(&sm.bar[i & (S - 1)]), (uint32_t)(i >> a.stage_shift) & 1u, nullptr);
    }
    __syncthreads();

    // ---- CTA partial -> slot r of the leader
    cluster_wait_acquire();                     // every CTA of the cluster has started
    {
        const uint32_t slot = smem_u32(part + (size_t)r * NG * (D + 2));
        const uint32_t dst = cluster_map(slot, 0);
        for (int x = threadIdx.x; x < NG * D; x += blockDim.x) {
            const int h = x / D, c = x % D;
            float M = kNegInf;
#pragma unroll
            for (int w = 0; w < W; ++w) M = fmaxf(M, sm.wm[w][h]);
            float L = 0.0f, O = 0.0f;
            if (M != kNegInf) {
#pragma unroll
                for (int w = 0; w < W; ++w) {
                    const float f = sm.wm[w][h] == kNegInf ? 0.0f : ex2_approx(sm.wm[w][h] - M);
                    L = fmaf(sm.wl[w][h], f, L);
                    O = fmaf(sm.wo[w][h][c], f, O);
                }
            }
            const uint32_t o = dst + (uint32_t)(h * (D + 2)) * 4u;
            cluster_st_f32(o + (uint32_t)(2 + c) * 4u, O);
            if (c == 0) {
                cluster_st_f32(o, M);
                cluster_st_f32(o + 4u, L);
            }
        }
    }
    cluster_arrive_release();
    cluster_wait_acquire();

    // ---- leader: merge the C partials, write o and lse
    if (r == 0) {
        if (threadIdx.x < 32) {
            // lane y holds partial y (C <= 32)
            const int y = threadIdx.x;
            for (int h = 0; h < NG; ++h) {
                float m = kNegInf, l = 0.0f;
                if (y < C) {
                    const float* p = part + ((size_t)y * NG + h) * (D + 2);
                    l = p[1];
                    m = l > 0.0f ? p[0] : kNegInf;
                }
                const float M = warp_max(m);
                const float w = m == kNegInf ? 0.0f : ex2_approx(m - M);
                const float L = warp_sum(l * w);
                if (y < C) sm.cw[y][h] = w;
                if (y == 0) {
                    sm.lsum[h] = L;
                    sm.lse2[h] = M + __log2f(L);
                    if (a.lse_out) a.lse_out[(size_t)b * a.Hq + hkv * NG + h] = (M + __log2f(L)) * kLn2;
                    if (a.lse2_ws) a.lse2_ws[unit * 8 + h] = M + __log2f(L);
                }
            }
        }
        __syncthreads();
        for (int x = threadIdx.x; x < NG * D; x += blockDim.x) {
            const int h = x / D, c = x % D;
            float acc = 0.0f;
            for (int y = 0; y < C; ++y) acc = fmaf(part[((size_t)y * NG + h) * (D + 2) + 2 + c], sm.cw[y][h], acc);
            stf(a.o, ((size_t)b * a.Hq + hkv * NG + h) * D + c, acc / sm.lsum[h], bf);
        }
    }

    // ---- DiffKV: every CTA adds the step's attention to its own ring tokens (MiKV
    // adds every token's in mikv_scores_kernel, after this launch)
    if (r == 0 && threadIdx.x == 0 && a.meta_ws) {
        a.meta_ws[unit * 4 + 0] = us.len;
        a.meta_ws[unit * 4 + 1] = us.start;
        a.meta_ws[unit * 4 + 2] = us.pos;
    }
    if (a.policy == KVQ_POLICY_DIFFKV && lg_unit) {
        if (r == 0 && threadIdx.x < NG)
            for (int y = 0; y < C; ++y)
                cluster_st_f32(cluster_map(smem_u32(&sm.lse2[threadIdx.x]), y), sm.lse2[threadIdx.x]);
        cluster_arrive_release();
        cluster_wait_acquire();
        add_scores<NG, D>(a, sm, unit, ir, n_local, lg_unit);
    }

    // ---- leader: MiniKV flush, counters
    if (r == 0) {
        const int cap = a.res_cap, len = us.len, start = us.start;
        __syncthreads();                        // C = 1: this CTA's own ring append is done
        bool flushed = false;
        if (a.policy == KVQ_POLICY_MINIKV && len + 1 == a.nr + a.G) {
            flushed = bf ? minikv_flush<__nv_bfloat16>(a, unit, start, us.cnt[0])
                         : minikv_flush<__half>(a, unit, start, us.cnt[0]);
            if (!flushed && threadIdx.x == 0) atomicOr(&g_status_decode, kDevCheck);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            if (flushed) {
                a.tier[0].count[unit] = us.cnt[0] + a.G;
                a.res_start[unit] = (start + a.G) % cap;
                a.res_len[unit] = len + 1 - a.G;
            } else {
                a.res_len[unit] = len + 1;
            }
            a.pos[unit] = us.pos + 1;
        }
    }
}


// ---- streamed decode: single heads, MiniKV format
//
// The units' items at full capacity form one static list: unit u owns items
// [u n_i, (u + 1) n_i) (its n_c tier chunks, then its n_r ring pieces), and
// CTA c takes the contiguous run [c per, (c + 1) per) of the list, as many CTAs
// as are resident at once.  Every SM then streams the same share of the layer
// whatever the batch, and a CTA's staging never drains between its units.  The
// issuing warp walks the run, skipping items past a unit's live counts, and
// publishes each requested item (unit, kind, index, tokens) beside its buffer;
// the other warps follow those records.  Per (CTA, unit) the CTA writes its
// partial state (max, sum, unnormalised output) to slot c + u of the
// workspace; a second launch merges each unit's partials and does the unit's
// end-of-step work (the new token into the ring, the MiniKV flush, counters).
struct StreamArgs {
    int n_c, n_r, n_i;           // tier chunks, ring pieces and items per unit at full capacity
    long long per, total;        // static items per CTA, items of all units
    float* part;                 // [ctas + units - 1][2 + 128] partial (max, sum, output) per (CTA, unit)
};

constexpr int kItChunk = 0, kItRing = 1, kItNone = 2, kItEnd = 3;

// Issuing warp (every lane; the warps take turns): requests the CTA's next item into
// buffer k % S and publishes its record; nothing but an end record once the run is done or
// a wait gave up.  Lanes 0..5 each copy one array of a tier chunk (at compile-time offsets
// of the format).  Not inlined: its registers stay out of the item loop's.
template <int GK, int CH>
__device__ __noinline__ void stream_issue(const DecodeArgs& a, const StreamArgs& s, Smem<1, 128>& sm,
                                          uint8_t* stage_base, int k, const uint8_t* cp_base, uint32_t cp_off,
                                          uint32_t cp_bpt) {
    constexpr uint32_t kSB = 256 / GK;
    const int lane = threadIdx.x & 31;
    int kind = kItEnd, u = 0, idx = 0, n = 0;
    if (lane == 0) {
        // the cursor: unit and item of the next static item, static items left in the run
        int uu = sm.wu, kk = sm.wk, rem = sm.fail ? 0 : sm.wrem;
        while (rem > 0) {
            if (uu != sm.cu) {
                const int raw = a.tier[0].count[uu], rl = a.res_len[uu], rs = a.res_start[uu];
                const int cnt = min(max(raw, 0), a.tier[0].cap), cap = a.res_cap;
                const int len = min(max(rl, 0), cap - 1), st = min(max(rs, 0), cap - 1);
                if (raw != cnt || rl != len || rs != st) atomicOr(&g_status_decode, kDevCheck);
                sm.cu = uu;
                sm.ccnt = cnt;
                sm.clen = len;
                sm.cstart = st;
                sm.cem = 0;
            }
            const int cu = uu, ck = kk;
            const bool last_of_unit = ck == s.n_i - 1 || rem == 1;
            --rem;
            if (++kk == s.n_i) {
                kk = 0;
                ++uu;
            }
            if (ck < s.n_c) {
                const int nn = min(CH, sm.ccnt - ck * CH);
                if (nn > 0) { kind = kItChunk; u = cu; idx = ck; n = nn; break; }
            } else {
                const int j0 = (ck - s.n_c) * kResItemS;
                const int nn = min(kResItemS, sm.clen + 1 - j0);
                if (nn > 0) { kind = kItRing; u = cu; idx = j0; n = nn; break; }
            }
            // a unit of the run with no live item still gets a record: its (empty) partial
            if (last_of_unit && !sm.cem) { kind = kItNone; u = cu; break; }
        }
        sm.wu = uu;
        sm.wk = kk;
        sm.wrem = rem;
        if (kind != kItEnd) sm.cem = 1;
        sm.meta[k & (a.stages - 1)] = make_int4(u, kind, idx, n);
    }
    kind = __shfl_sync(0xffffffffu, kind, 0);
    if (kind == kItEnd) return;
    u = __shfl_sync(0xffffffffu, u, 0);
    idx = __shfl_sync(0xffffffffu, idx, 0);
    n = __shfl_sync(0xffffffffu, n, 0);
    const int sb = k & (a.stages - 1);
    const uint32_t bar = smem_u32(&sm.bar[sb]);
    const uint32_t dst = smem_u32(stage_base) + (uint32_t)sb * a.stage_bytes;
    // failure-detection check: the first CTA withholds its first item's copies
    const bool withhold = a.withhold_unit >= 0 && blockIdx.x == 0 && k == 0 && kind != kItNone;
    if (kind == kItChunk) {
        const int np = (n + 31) & ~31;
        if (lane == 0 && !withhold) mbar_expect_tx(bar, (64u + 4u * kSB) * (uint32_t)np);
        __syncwarp();
        if (lane < 6 && !withhold)
            bulk_load(dst + cp_off * (uint32_t)np,
                      cp_base + ((size_t)u * a.tier[0].cap + (size_t)idx * CH) * cp_bpt, cp_bpt * (uint32_t)np, bar);
    } else if (lane == 0 && !withhold) {
        if (kind == kItRing)
            stage_residual(a, (size_t)u, sm.clen, sm.cstart, idx, n, 128, stage_base + (size_t)sb * a.stage_bytes, bar);
        else
            mbar_arrive(bar);                            // no bytes: the buffer's phase completes at once
    }
    if (lane == 0) sm.issued = k + 1;
}

// Every warp is done with item i: warp i mod W (the turns spread the issuing work) requests
// item i + S into its buffer.
template <int GK, int CH>
__device__ __forceinline__ void stream_release(const DecodeArgs& a, const StreamArgs& s, Smem<1, 128>& sm,
                                               uint8_t* stage_base, int i, const uint8_t* cp_base,
                                               uint32_t cp_off, uint32_t cp_bpt) {
    __syncthreads();
    if ((threadIdx.x >> 5) == (i & (Cfg<1>::W - 1)))
        stream_issue<GK, CH>(a, s, sm, stage_base, i + a.stages, cp_base, cp_off, cp_bpt);
}

// Grid = (CTAs): CTA c streams the static items [c per, min((c + 1) per, total)); a tier
// chunk is CH tokens (128 or 256: each warp takes 32 tokens of each 128).
template <int GK, int CH>
__global__ void __launch_bounds__(Cfg<1>::kThreads, Cfg<1>::MINB) decode_stream_kernel(DecodeArgs a, StreamArgs s) {
    constexpr int D = 128, W = Cfg<1>::W, TPW = Cfg<1>::TPW;
    constexpr uint32_t kSB = 256 / GK;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem<1, D>& sm = *reinterpret_cast<Smem<1, D>*>(smem_raw);
    uint8_t* stage_base = smem_raw + a.stage_off;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool bf = a.bf16 != 0;
    // lanes 0..5 of the issuing warp copy one array of a tier chunk each: unit u's chunk j
    // starts (u cap + CH j) bytes_per_token into the array
    const TierArgs& ta = a.tier[0];
    const uint8_t* cp_base = nullptr;
    uint32_t cp_off = 0u, cp_bpt = 0u;
    switch (lane) {
        case 0: cp_base = reinterpret_cast<const uint8_t*>(ta.k_codes); cp_off = 0; cp_bpt = 32; break;
        case 1: cp_base = reinterpret_cast<const uint8_t*>(ta.k_scale); cp_off = 32; cp_bpt = kSB; break;
        case 2: cp_base = reinterpret_cast<const uint8_t*>(ta.k_zero); cp_off = 32 + kSB; cp_bpt = kSB; break;
        case 3: cp_base = reinterpret_cast<const uint8_t*>(ta.v_codes); cp_off = 32 + 2 * kSB; cp_bpt = 32; break;
        case 4: cp_base = reinterpret_cast<const uint8_t*>(ta.v_scale); cp_off = 64 + 2 * kSB; cp_bpt = kSB; break;
        case 5: cp_base = reinterpret_cast<const uint8_t*>(ta.v_zero); cp_off = 64 + 3 * kSB; cp_bpt = kSB; break;
        default: break;
    }
    grid_launch_dependents();                            // the merge launch may start as CTAs retire
    if (threadIdx.x == 0) {
        for (int st = 0; st < a.stages; ++st) mbar_init(smem_u32(&sm.bar[st]), 1);
        sm.fail = 0;
        sm.issued = 0;
        const long long g0 = (long long)blockIdx.x * s.per;
        sm.wu = (int)(g0 / s.n_i);
        sm.wk = (int)(g0 - (long long)sm.wu * s.n_i);
        sm.wrem = (int)min(s.per, s.total - g0);
        sm.cu = -1;
        sm.cem = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0)
        for (int k = 0; k < a.stages; ++k) stream_issue<GK, CH>(a, s, sm, stage_base, k, cp_base, cp_off, cp_bpt);
    __syncthreads();                                     // the first S records are visible

    // A record is written when its item is requested, at least one CTA barrier before any
    // warp reads it (S >= 2), so every warp takes the same path through the run.
    bool ok = true;
    int i = 0;
    for (;;) {
        const int4 m0 = sm.meta[i & (a.stages - 1)];
        if (m0.y == kItEnd) break;
        const int u = m0.x;
        // the unit's query (base-2 logits; one query head per KV head) and fresh warp states
        for (int x = threadIdx.x; x < D; x += blockDim.x) sm.q[0][x] = ldf(a.q, (size_t)u * D + x, bf) * a.scale_log2;
        for (int x = threadIdx.x; x < W; x += blockDim.x) {
            sm.wm[x][0] = kNegInf;
            sm.wl[x][0] = 0.0f;
        }
        for (int x = threadIdx.x; x < W * D; x += blockDim.x) (&sm.wo[0][0][0])[x] = 0.0f;
        __syncthreads();
        int4 m = m0;
        if (m.y == kItChunk) {
            const Mk1Ctx<GK> x = mk1_ctx<GK>(a, sm);
            Mk1Acc<GK> acc;
            mk1_acc_init(acc);
            do {
                ok = wait_item(a, sm, i, ok);
                const int n = m.w;
                if constexpr (CH == kSub) {
                    const int tl = warp * TPW;
                    if (ok && tl < n)
                        mk1_item<GK>(mk1_view<GK>((n + 31) & ~31, item_buf(a, stage_base, i)), tl, min(TPW, n - tl), x, acc);
                } else if (ok) {
                    const uint8_t* buf = item_buf(a, stage_base, i);
#pragma unroll 1
                    for (int h = 0; h < CH / kSub; ++h) {
                        const int tl = h * kSub + warp * TPW;
                        if (tl < n) mk1_item<GK>(mk1_view<GK>((n + 31) & ~31, buf), tl, min(TPW, n - tl), x, acc);
                    }
                }
                stream_release<GK, CH>(a, s, sm, stage_base, i, cp_base, cp_off, cp_bpt);
                m = sm.meta[++i & (a.stages - 1)];
            } while (m.y == kItChunk && m.x == u);
            mk1_flush<GK>(acc, sm);
        }
        if (m.y == kItRing && m.x == u) {
            WarpAcc<1, D / 32> racc;
            acc_init(racc);
            do {
                ok = wait_item(a, sm, i, ok);
                constexpr int RPS = kResItemS / W;       // ring rows per warp and item
                const int n = m.w, w0 = warp * RPS;
                if (ok && w0 < n) {
                    const uint8_t* buf = item_buf(a, stage_base, i);
                    const uint16_t* rk = reinterpret_cast<const uint16_t*>(buf);
                    const uint16_t* rv = reinterpret_cast<const uint16_t*>(buf + a16((uint32_t)n * D * 2));
                    residual_rows<1, D, RPS>(sm, rk + (size_t)w0 * D, rv + (size_t)w0 * D, min(RPS, n - w0), bf,
                                             racc, nullptr, a.slots);
                }
                stream_release<GK, CH>(a, s, sm, stage_base, i, cp_base, cp_off, cp_bpt);
                m = sm.meta[++i & (a.stages - 1)];
            } while (m.y == kItRing && m.x == u);
            flush_lane_values<1, D>(racc, sm);
        }
        if (m.y == kItNone && m.x == u) {                // nothing staged: its barrier completed at once
            stream_release<GK, CH>(a, s, sm, stage_base, i, cp_base, cp_off, cp_bpt);
            ++i;
        }
        __syncthreads();                                 // every warp's state is in shared memory
        // the partial of (this CTA, u): slot blockIdx.x + u
        float* pp = s.part + ((size_t)blockIdx.x + (size_t)u) * (D + 2);
        for (int c = threadIdx.x; c < D; c += blockDim.x) {
            float M = kNegInf;
#pragma unroll
            for (int w = 0; w < W; ++w) M = fmaxf(M, sm.wm[w][0]);
            float L = 0.0f, O = 0.0f;
            if (M != kNegInf) {
#pragma unroll
                for (int w = 0; w < W; ++w) {
                    const float f = sm.wm[w][0] == kNegInf ? 0.0f : ex2_approx(sm.wm[w][0] - M);
                    L = fmaf(sm.wl[w][0], f, L);
                    O = fmaf(sm.wo[w][0][c], f, O);
                }
            }
            pp[2 + c] = O;
            if (c == 0) {
                pp[0] = M;
                pp[1] = L;
            }
        }
        __syncthreads();                                 // before the next unit's query and states
    }
    __syncthreads();
    if (sm.fail && threadIdx.x == 0) {
        atomicOr(&g_status_decode, kDevTimeout);
        // let every copy still in flight land before the buffers go away
        const int S = a.stages, n = sm.issued;
        for (int k = max(0, n - S); k < n; ++k)
            (void)mbar_wait(smem_u32(&sm.bar[k & (S - 1)]), (uint32_t)(k >> a.stage_shift) & 1u, nullptr);
    }
}

// Grid = (units), one thread per channel: the unit's partials (slots c + u of the CTAs whose
// runs meet the unit) merged into o and lse, then its end-of-step work as the cluster
// leader does it.  Launched as a programmatic dependent of the streamed launch: what does
// not depend on it is read before the grid dependency wait.
__global__ void __launch_bounds__(128) decode_stream_finalize(DecodeArgs a, StreamArgs s) {
    constexpr int D = 128;
    const int u = blockIdx.x, c = threadIdx.x;
    const bool bf = a.bf16 != 0;
    const int raw = a.tier[0].count[u], rl = a.res_len[u], rs = a.res_start[u], ps = a.pos[u];
    const float kn = ldf(a.k_new, (size_t)u * D + c, bf), vn = ldf(a.v_new, (size_t)u * D + c, bf);
    const long long first = (long long)u * s.n_i;
    const int c0 = (int)(first / s.per), nseg = (int)((first + s.n_i - 1) / s.per) - c0 + 1;
    const float* part = s.part + ((size_t)c0 + (size_t)u) * (D + 2);   // slot c + u, c = c0 .. c0 + nseg - 1
    grid_dependency_wait();
    // online merge of the partials (empty ones have sum 0)
    float M = kNegInf, L = 0.0f, O = 0.0f;
    for (int y = 0; y < nseg; ++y) {
        const float* p = part + (size_t)y * (D + 2);
        const float m = p[0], l = p[1], o = p[2 + c];
        if (!(l > 0.0f)) continue;
        if (m > M) {
            const float f = M == kNegInf ? 0.0f : ex2_approx(M - m);
            L = fmaf(L, f, l);
            O = fmaf(O, f, o);
            M = m;
        } else {
            const float w = ex2_approx(m - M);
            L = fmaf(l, w, L);
            O = fmaf(o, w, O);
        }
    }
    stf(a.o, (size_t)u * D + c, O / L, bf);
    if (c == 0 && a.lse_out) a.lse_out[u] = (M + __log2f(L)) * kLn2;
    // the new token joins the ring, then the MiniKV flush when the ring is full
    const int cap = a.res_cap, cnt = min(max(raw, 0), a.tier[0].cap);
    const int len = min(max(rl, 0), cap - 1), start = min(max(rs, 0), cap - 1);
    const size_t slot = (size_t)u * cap + (start + len) % cap;
    stf(a.res_k, slot * D + c, kn, bf);
    stf(a.res_v, slot * D + c, vn, bf);
    if (c == 0) a.res_token_id[slot] = ps;
    bool flushed = false;
    if (len + 1 == a.nr + a.G) {                         // the same for every thread of the block
        __syncthreads();                                 // the new row is in the ring
        flushed = bf ? minikv_flush<__nv_bfloat16>(a, (size_t)u, start, cnt)
                     : minikv_flush<__half>(a, (size_t)u, start, cnt);
        if (!flushed && c == 0) atomicOr(&g_status_decode, kDevCheck);
        __syncthreads();
    }
    if (c == 0) {
        if (flushed) {
            a.tier[0].count[u] = cnt + a.G;
            a.res_start[u] = (start + a.G) % cap;
            a.res_len[u] = len + 1 - a.G;
        } else {
            a.res_len[u] = len + 1;
        }
        a.pos[u] = ps + 1;
    }
}

struct WsLayout {
    int slots;
    size_t logits, lse2, meta, part, total;
};

WsLayout ws_layout(const kvq_cache& c) {
    WsLayout w{};
    const int units = c.B * c.Hkv, g = c.Hq / c.Hkv;
    int slots = 0;
    for (int t = 0; t < c.n_tiers; ++t) slots += c.tier[t].cap;
    slots += c.res_cap;
    w.slots = slots;
    w.logits = 0;
    w.total = c.policy != KVQ_POLICY_MINIKV ? (size_t)units * g * slots * sizeof(float) : 0;
    // MiniKV with one query head per KV head (streamed decode): a partial per (CTA, unit)
    if (c.policy == KVQ_POLICY_MINIKV && g == 1 && c.D == 128) {
        w.part = 0;
        w.total = (size_t)(kStreamMaxCtas + units) * (c.D + 2) * sizeof(float);
    }
    if (c.policy == KVQ_POLICY_MIKV) {
        w.lse2 = (w.total + 255) & ~(size_t)255;
        w.meta = w.lse2 + (size_t)units * 8 * sizeof(float);
        w.total = w.meta + (size_t)units * 4 * sizeof(int32_t);
    }
    return w;
}

// Items of a unit at full capacity (an upper bound of the live count).
int items_bound(const kvq_cache& c) {
    int n = 0;
    for (int t = 0; t < c.n_tiers; ++t) n += (c.tier[t].cap + kSub - 1) / kSub;
    return n + (c.res_cap + kResItem - 1) / kResItem;
}

// Streamed decode (single heads, MiniKV format): as many CTAs as are resident at once, at
// most kStreamMaxCtas; runs shorter than kStreamMinItems items per CTA take the cluster path.

// The streamed launch's shape for a cache (device-dependent: resident CTAs per SM).
struct StreamPlan {
    bool used;                   // false: the cluster path
    StreamArgs sa;
    int ctas, S;
    uint32_t stage, sm_bytes, qf_bytes, smem;
};

template <int GK>
cudaError_t stream_plan(const kvq_cache& c, int units, StreamPlan& p) {
    constexpr int D = 128, CH = kStreamChunk<GK>;
    p = StreamPlan{};
    StreamArgs& sa = p.sa;
    sa.n_c = (c.tier[0].cap + CH - 1) / CH;
    sa.n_r = (c.res_cap + kResItemS - 1) / kResItemS;
    sa.n_i = sa.n_c + sa.n_r;
    sa.total = (long long)units * sa.n_i;
    uint32_t stage = std::max(tier_stage_sizes(KVQ_AXIS_CHANNEL, 2, 2, CH, D, GK).total(),
                              2u * a16((uint32_t)kResItemS * D * 2));
    p.stage = (stage + 127u) & ~127u;
    p.sm_bytes = (uint32_t)((sizeof(Smem<1, D>) + 127) & ~(size_t)127);
    p.qf_bytes = (uint32_t)Cfg<1>::W * mk1_qf_warp_bytes<GK>();
    constexpr uint32_t kSmemLimit = 227u * 1024u;
    auto smem_for = [&](int S) { return p.sm_bytes + p.qf_bytes + (uint32_t)S * p.stage; };
    auto kern = decode_stream_kernel<GK, CH>;
    // resident CTAs per SM with 2 and 4 staging buffers, and the SM count, per device
    constexpr int kDevs = 16;
    static int per_sm[kDevs][2], sms[kDevs];
    static bool known[kDevs] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kDevs) return cudaSuccess;             // not used: the cluster path
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!known[dev]) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)std::min(smem_for(kMaxStages), kSmemLimit));
            if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
            for (int k = 0; k < 2 && e == cudaSuccess; ++k) {
                per_sm[dev][k] = 0;
                if (smem_for(2 << k) <= kSmemLimit)
                    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm[dev][k], kern, Cfg<1>::kThreads,
                                                                      smem_for(2 << k));
            }
            if (e != cudaSuccess) return e;
            known[dev] = true;
        }
    }
    // four buffers where they cost no resident CTA
    p.S = per_sm[dev][1] >= per_sm[dev][0] && per_sm[dev][1] > 0 ? 4 : 2;
    const long long resident = (long long)per_sm[dev][p.S == 4 ? 1 : 0] * sms[dev];
    int ctas = (int)std::min<long long>(resident, kStreamMaxCtas);
    if (ctas < 1 || sa.total < (long long)kStreamMinItems * ctas) return cudaSuccess;
    sa.per = (sa.total + ctas - 1) / ctas;
    p.ctas = (int)((sa.total + sa.per - 1) / sa.per);
    p.smem = smem_for(p.S);
    p.used = true;
    return cudaSuccess;
}

template <int GK>
cudaError_t launch_stream(DecodeArgs& a, const kvq_cache& c, int units, cudaStream_t s, bool& used) {
    constexpr int D = 128;
    used = false;
    StreamPlan p;
    cudaError_t e = stream_plan<GK>(c, units, p);
    if (e != cudaSuccess || !p.used) return e;
    p.sa.part = a.stream_part;
    a.cluster = 1;
    a.stages = p.S;
    a.stage_shift = p.S == 4 ? 2 : 1;
    a.stage_bytes = p.stage;
    a.qf_off = p.sm_bytes;
    a.part_off = p.sm_bytes + p.qf_bytes;
    a.stage_off = p.sm_bytes + p.qf_bytes;
    decode_stream_kernel<GK, kStreamChunk<GK>><<<p.ctas, Cfg<1>::kThreads, p.smem, s>>>(a, p.sa);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)units);
    cfg.blockDim = dim3(D);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    used = true;
    return cudaLaunchKernelEx(&cfg, decode_stream_finalize, a, p.sa);
}

template <int NG, int D, int FAM>
cudaError_t launch_typed(DecodeArgs& a, const kvq_cache& c, int units, cudaStream_t s) {
    if constexpr (NG == 1 && D == 128 && FAM == 1) {
        if (c.policy == KVQ_POLICY_MINIKV && a.stream_part) {
            bool used = false;
            const cudaError_t e = c.G == 16 ? launch_stream<16>(a, c, units, s, used)
                                            : launch_stream<32>(a, c, units, s, used);
            if (e != cudaSuccess || used) return e;
        }
    }
    uint32_t stage = 2u * a16((uint32_t)kResItem * D * 2);
    for (int t = 0; t < c.n_tiers; ++t)
        stage = std::max(stage, tier_stage_sizes(c.tier[t].k_axis, c.tier[t].k_bits, c.tier[t].v_bits,
                                                 kSub, D, c.G).total());
    stage = (stage + 127u) & ~127u;
    const uint32_t sm_bytes = (uint32_t)((sizeof(Smem<NG, D>) + 127) & ~(size_t)127);
    // per-channel keys on the tensor cores: each warp's query x scale rows
    bool has_channel = false;
    for (int t = 0; t < c.n_tiers; ++t) has_channel |= c.tier[t].k_axis == KVQ_AXIS_CHANNEL;
    // (single heads: query pieces and, with G = 16, the value-group products of each warp)
    const uint32_t qf_bytes = (has_channel && D == 128 && NG <= 4)
                                  ? (NG == 1 ? (uint32_t)Cfg<NG>::W * (c.G == 16 ? mk1_qf_warp_bytes<16>()
                                                                                  : mk1_qf_warp_bytes<32>())
                                             : (uint32_t)(Cfg<NG>::W * 2 * NG * 128 * sizeof(uint16_t)))
                                  : 0u;
    const uint32_t slot_bytes = (uint32_t)(NG * (D + 2) * sizeof(float));
    auto smem_for = [&](int C, int S) {
        return sm_bytes + qf_bytes + ((C * slot_bytes + 127u) & ~127u) + (uint32_t)S * stage;
    };
    constexpr uint32_t kSmemLimit = 227u * 1024u;
    int cmax = kMaxCluster;
    while (cmax > 1 && (uint32_t)cmax * slot_bytes > 32u * 1024u) cmax >>= 1;

    auto kern = decode_kernel<NG, D, FAM>;
    static bool attr_done = false, wide_ok = false;
    if (!attr_done) {
        const uint32_t qf_max = NG == 1 ? (uint32_t)Cfg<NG>::W * mk1_qf_warp_bytes<16>()
                                        : (NG <= 4 ? (uint32_t)(Cfg<NG>::W * 2 * NG * 128 * sizeof(uint16_t)) : 0u);
        cudaError_t e = cudaFuncSetAttribute(
            kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
            (int)std::min(smem_for(kMaxCluster, kMaxStages) - qf_bytes + qf_max, kSmemLimit));
        if (e != cudaSuccess) return e;
        // clusters above the portable 8 CTAs, where the device allows them
        wide_ok = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
        if (!wide_ok) (void)cudaGetLastError();
        attr_done = true;
    }
    if (!wide_ok) cmax = std::min(cmax, 8);
    // CTAs per unit (a power of two, at most cmax and at most the items): as
    // many as one wave of resident CTAs holds (small caches: the shortest
    // chain per CTA), or, when the units alone fill the GPU, the most that
    // still leave every CTA kMinItemsPerCta items (large caches: enough
    // clusters to smooth the wave tail, few enough that each CTA's fixed
    // cost stays small against its stream).
    // the choice per cache shape, remembered (a model's layers differ only in capacity; the
    // first call of each shape queries occupancy, later ones -- e.g. under stream capture --
    // only look it up)
    constexpr int kShapes = 64;
    static int known[kShapes][8];
    static int n_known = 0;
    static std::mutex known_mu;
    std::lock_guard<std::mutex> lock(known_mu);
    const int items = items_bound(c);
    const int key[6] = {units, items, (int)stage, c.n_tiers, (int)qf_bytes, c.policy};
    int C = 0, S = 2;
    for (int i = 0; i < n_known && !C; ++i)
        if (std::equal(key, key + 6, known[i])) {
            C = known[i][6];
            S = known[i][7];
        }
    if (!C) {
        int dev = 0, sms = 0, per_sm = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Cfg<NG>::kThreads, smem_for(cmax, 2));
        if (e != cudaSuccess) return e;
        const long resident = (long)std::max(per_sm, 1) * sms;
        int c_fill = 1, c_items = 1;
        while (c_fill * 2 <= std::min(cmax, items) && (long)units * c_fill * 2 <= resident) c_fill *= 2;
        const int min_items = c.policy == KVQ_POLICY_MIKV ? kMinItemsPerCtaMikv : kMinItemsPerCta;
        while (c_items * 2 <= std::min(cmax, items) && (items + 2 * c_items - 1) / (2 * c_items) >= min_items)
            c_items *= 2;
        C = std::max(c_fill, c_items);
        for (; C > 1; C >>= 1) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = (unsigned)C;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3((unsigned)C, (unsigned)units);
            cfg.blockDim = dim3(Cfg<NG>::kThreads);
            cfg.dynamicSmemBytes = smem_for(C, 2);
            cfg.attrs = at;
            cfg.numAttrs = 1;
            int ncl = 0;
            if (cudaOccupancyMaxActiveClusters(&ncl, kern, &cfg) == cudaSuccess && ncl > 0) break;
            (void)cudaGetLastError();
        }
        // staging buffers: as many as fit without costing a resident CTA
        int occ2 = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ2, kern, Cfg<NG>::kThreads, smem_for(C, 2)) != cudaSuccess)
            (void)cudaGetLastError();
        for (int s2 = kMaxStages; s2 > 2; s2 >>= 1) {
            int o = 0;
            if (smem_for(C, s2) > kSmemLimit) continue;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, Cfg<NG>::kThreads, smem_for(C, s2)) != cudaSuccess) {
                (void)cudaGetLastError();
                continue;
            }
            if (o >= occ2) {
                S = s2;
                break;
            }
        }
        const int slot = n_known < kShapes ? n_known++ : (int)((unsigned)items % kShapes);
        std::copy(key, key + 6, known[slot]);
        known[slot][6] = C;
        known[slot][7] = S;
    }
    a.cluster = C;
    a.stages = S;
    a.stage_shift = S == 4 ? 2 : 1;
    a.stage_bytes = stage;
    a.qf_off = sm_bytes;
    a.part_off = sm_bytes + qf_bytes;
    a.stage_off = a.part_off + ((C * slot_bytes + 127u) & ~127u);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)C;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)C, (unsigned)units);
    cfg.blockDim = dim3(Cfg<NG>::kThreads);
    cfg.dynamicSmemBytes = smem_for(C, S);
    cfg.stream = s;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

size_t decode_workspace_bytes(const kvq_cache& c) { return ws_layout(c).total; }

int decode_launches(const kvq_cache& c) {
    const int units = c.B * c.Hkv;
    int n = c.policy == KVQ_POLICY_MIKV ? 2 : 1;               // MiKV: the score kernel after the step
    if (c.policy == KVQ_POLICY_MINIKV && c.Hq == c.Hkv && c.D == 128) {
        StreamPlan p;
        const cudaError_t e = c.G == 16 ? stream_plan<16>(c, units, p) : stream_plan<32>(c, units, p);
        if (e != cudaSuccess) return -1;
        if (p.used) n = 2;                                     // streamed: the merge launch after it
    }
    return n;
}

namespace {
std::atomic<int> g_withhold_copy{0};
}  // namespace

void set_withhold_copy(int on) { g_withhold_copy.store(on ? 1 : 0); }

cudaError_t launch_decode(const void* q, const void* k_new, const void* v_new, const kvq_cache& c,
                          float sm_scale, void* o, float* lse_out, void* ws, cudaStream_t s) {
    const WsLayout w = ws_layout(c);
    const int units = c.B * c.Hkv;
    if (units > 65535) return cudaErrorInvalidConfiguration;
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
    a.nr = c.nr;
    a.withhold_unit = g_withhold_copy.load() ? 0 : -1;
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
        ta.page_table = ct.page_table;
        ta.max_pages = ct.max_pages;
        ta.n_pages = ct.n_pages;
        ta.slot_base = slot;
        slot += ct.cap;
    }
    a.res_k = c.res_k;
    a.res_v = c.res_v;
    a.res_token_id = c.res_token_id;
    a.res_start = c.res_start;
    a.res_len = c.res_len;
    a.res_cap = c.res_cap;
    a.res_slot_base = slot;
    a.pos = c.seq_len;
    a.win_acc = c.win_acc;
    a.cum_score = c.cum_score;
    a.score_cap = c.score_cap;
    a.scale_log2 = sm_scale * kLog2e;
    a.slots = w.slots;
    a.logits = c.policy != KVQ_POLICY_MINIKV ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + w.logits)
                                             : nullptr;
    a.lse2_ws = c.policy == KVQ_POLICY_MIKV ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + w.lse2) : nullptr;
    a.meta_ws = c.policy == KVQ_POLICY_MIKV ? reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + w.meta) : nullptr;
    a.stream_part = c.policy == KVQ_POLICY_MINIKV && a.g == 1 && c.D == 128 && ws
                        ? reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + w.part)
                        : nullptr;
    bool channel_only = true;
    for (int t = 0; t < c.n_tiers; ++t) channel_only &= c.tier[t].k_axis == KVQ_AXIS_CHANNEL;
    if (c.D == 64) return a.g == 1 ? launch_typed<1, 64, 1>(a, c, units, s) : cudaErrorInvalidConfiguration;
    if (c.D != 128) return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaErrorInvalidConfiguration;
    switch (a.g * 2 + (channel_only ? 0 : 1)) {
        case 2: e = launch_typed<1, 128, 1>(a, c, units, s); break;
        case 3: e = launch_typed<1, 128, 3>(a, c, units, s); break;
        case 4: e = launch_typed<2, 128, 1>(a, c, units, s); break;
        case 5: e = launch_typed<2, 128, 3>(a, c, units, s); break;
        case 8: e = launch_typed<4, 128, 1>(a, c, units, s); break;
        case 9: e = launch_typed<4, 128, 3>(a, c, units, s); break;
        case 10: e = launch_typed<5, 128, 1>(a, c, units, s); break;
        case 11: e = launch_typed<5, 128, 3>(a, c, units, s); break;
        case 16: e = launch_typed<8, 128, 1>(a, c, units, s); break;
        case 17: e = launch_typed<8, 128, 3>(a, c, units, s); break;
    }
    if (e != cudaSuccess || c.policy != KVQ_POLICY_MIKV) return e;
    // MiKV: every token's score, once the step's lse is known
    ScoreArgs sa{};
    sa.g = a.g;
    sa.n_tiers = c.n_tiers;
    sa.slots = w.slots;
    sa.res_cap = c.res_cap;
    sa.res_slot_base = a.res_slot_base;
    sa.score_cap = c.score_cap;
    for (int t = 0; t < c.n_tiers; ++t) {
        sa.token_id[t] = c.tier[t].token_id;
        sa.count[t] = c.tier[t].count;
        sa.cap[t] = c.tier[t].cap;
        sa.slot_base[t] = a.tier[t].slot_base;
    }
    sa.res_token_id = c.res_token_id;
    sa.logits = a.logits;
    sa.lse2 = a.lse2_ws;
    sa.meta = a.meta_ws;
    sa.cum_score = c.cum_score;
    const dim3 grid((unsigned)((w.slots + 255) / 256), (unsigned)units);
    mikv_scores_kernel<<<grid, 256, 0, s>>>(sa);
    return cudaGetLastError();
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
