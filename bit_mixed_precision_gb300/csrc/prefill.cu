// prefill_attn_scores: the two-pass prefill of MiniKV (review page, referee
// minor comment 2 on section 3.2 -- pass 1 follows FlashAttention's online
// softmax; Figure 4 caption -- two-pass kernel parallelism; verdict JSON
// key_machinery -- output plus column-wise cumulative attention scores with
// memory linear in the sequence length).
//
// GB300 design (tcgen05 + TMEM + TMA, one CTA per 128-row tile):
//   pass 1 (row-parallel): CTA = (batch*query head, query tile of 128).
//     warp 4 = TMA producer (Q once, K/V tiles double-buffered),
//     warp 5 = MMA issuer: S = Q K^T into one of two TMEM S buffers, then
//              O += P V into the TMEM O accumulator,
//     warps 0-3 = softmax: thread r owns query row r (TMEM lane r), reads
//              its S row, keeps the running max/sum, writes P (fp16) back
//              over the first half of the same S buffer (the P.V MMA reads
//              its A operand from TMEM, so P is double-buffered with S and
//              the next tile's P never waits for this tile's P.V), rescales
//              O only when its max grew by more than 2^8 (exact: the final
//              division uses the same stale max), and finally writes O / l
//              and lse.
//   pass 2 (column-parallel): CTA = (batch*query head, key tile of 128),
//     loops over the query tiles at or below the diagonal; S^T = K Q^T in
//     TMEM; thread r owns key r and sums exp(S - lse_i) over queries, so
//     column sums stay in registers (no atomics, no T x T buffer).
// Every mbarrier wait is bounded (2 s, or at once after another warp gave
// up); a timed-out CTA drains its copies and MMAs, frees TMEM and records
// KVQ_ETIMEOUT in the device status word.
#include <mutex>

#include <algorithm>

#include "kvq_common.cuh"
#include "kvq_internal.h"

namespace kvq {

KVQ_DEFINE_STATUS(prefill)

namespace {

constexpr int kTile = 128;                 // rows per tile (queries or keys)
constexpr uint32_t kHalfBytes = 128 * 128;       // one 128-row x 64-column 128B-swizzled half
constexpr int kBN = 64;                          // keys per K/V tile of pass 1
constexpr uint32_t kKVHalf = kBN * 128;          // one 64-row x 64-column swizzled half
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.0f;
// pass 2: two warpgroups sum the exponentials (each half of a tile's query columns), then
// one TMA warp and one MMA warp
constexpr int kP2Threads = 320;
constexpr long long kL2OrderBytes = 128ll << 20;  // about L2 (129 MB): the prefill launch order's threshold

// Shared memory maps (offsets from a 1024-aligned base) for head dim D.
template <int D> struct Layout {
    static constexpr uint32_t kTileBytes = kTile * D * 2;      // D/64 halves
    static constexpr uint32_t kKVBytes = kBN * D * 2;          // pass-1 K or V tile, D/64 halves
    // pass 1 (about 96 KB at D = 128: two CTAs per SM; P lives in TMEM)
    static constexpr uint32_t P1_Q = 0;
    static constexpr uint32_t P1_K = P1_Q + kTileBytes;        // 2 stages
    static constexpr uint32_t P1_V = P1_K + 2 * kKVBytes;      // 2 stages
    static constexpr uint32_t P1_BAR = P1_V + 2 * kKVBytes;
    // no alignment slack: two CTAs must fit one SM, so the kernel requires (and
    // checks) a 1024-aligned dynamic shared memory base
    static constexpr uint32_t P1_SMEM = P1_BAR + 256;
    // pass 2
    static constexpr uint32_t P2_K = 0;
    static constexpr uint32_t P2_Q = P2_K + kTileBytes;        // 2 stages
    static constexpr uint32_t P2_LSE = P2_Q + 2 * kTileBytes;  // 2 x 128 floats
    static constexpr uint32_t P2_RED = P2_LSE + 2 * kTile * 4; // the second warpgroup's sums and flags
    static constexpr uint32_t P2_BAR = P2_RED + 2 * kTile * 4;
    static constexpr uint32_t P2_SMEM = P2_BAR + 256 + 1024;
};

// pass 1: K/V tiles prefetched into L2 this far ahead (measured: 1 and 4 equal at 4k-token
// prompts; at 16k tokens 1 is 10 % faster than 4, whose prefetches crowd L2)
constexpr int kKVPrefetch = 1;
enum P1Bar { B_Q = 0, B_KF = 1, B_VF = 3, B_KVE = 5, B_SF = 7, B_SCONS = 8, B_SFREE = 9, B_PF = 11, B_OD = 13,
             B_DRAIN = 14, B_VC = 15, P1_NBAR = 17 };
enum P2Bar { C_KF = 0, C_QF = 1, C_QE = 3, C_SF = 5, C_SFREE = 7, C_DRAIN = 9, C_LSE = 10,
             P2_NBAR = 12 };

template <typename T> struct Pack2;
template <> struct Pack2<__half> {
    static __device__ __forceinline__ uint32_t pack(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
};
template <> struct Pack2<__nv_bfloat16> {
    static __device__ __forceinline__ uint32_t pack(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
};

// Bounded wait whose outcome is the same for every lane of the warp, so that
// the warp-collective tcgen05.ld/st after it stay convergent.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag)) != 0;
}

__device__ __forceinline__ void give_up(volatile int* abort_flag) {
    *abort_flag = 1;
    atomicOr(&g_status_prefill, kDevTimeout);
}

// K-major operand (rows x 128 elements as two 128B-swizzled 64-column halves):
// descriptor of the 16-element K slice kk (0..7).
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk, uint32_t half = kHalfBytes) {
    return sdesc_sw128(tile + (uint32_t)(kk >> 2) * half + (uint32_t)(kk & 3) * 32u, 16u,
                       1024u);
}

// MN-major operand (128 K-rows of 128 N-elements, two 64-column halves):
// descriptor of K rows 16*kk .. 16*kk+15.  LBO = stride between the N
// halves, SBO = stride between groups of 8 K rows.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile, int kk, uint32_t half = kHalfBytes) {
    return sdesc_sw128(tile + (uint32_t)kk * 16u * 128u, half, 1024u);
}

template <typename T, int AB, int D>
__global__ void __launch_bounds__(192, 2)
    prefill_pass1_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                         const __grid_constant__ CUtensorMap tv, T* __restrict__ o,
                         float* __restrict__ lse, int T_len, int Hq, int Hkv, int n_qt,
                         float scale_log2, int tile_fast) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    if (raw & 1023u) {                                  // layout assumption broken: do nothing
        if (threadIdx.x == 0) atomicOr(&g_status_prefill, kDevCheck);
        return;
    }
    const uint32_t base = raw;
    uint8_t* gbase = smem_raw;
    using Lay = Layout<D>;
    constexpr uint32_t kTileBytes = Lay::kTileBytes;
    constexpr uint32_t kKVBytes = Lay::kKVBytes;
    constexpr int kHalves = D / 64;
    const uint32_t sQ = base + Lay::P1_Q, sK = base + Lay::P1_K, sV = base + Lay::P1_V;
    const uint32_t bar0 = base + Lay::P1_BAR;
    auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + Lay::P1_BAR + 8 * P1_NBAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + Lay::P1_BAR + 8 * P1_NBAR + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // tile_fast: blockIdx.x runs over the head's query tiles, blockIdx.y over heads (the CTAs
    // resident together then read a few heads' K/V and reuse it in L2)
    const int bh = tile_fast ? (int)blockIdx.y : (int)blockIdx.x;
    const int qt = n_qt - 1 - (tile_fast ? (int)blockIdx.x : (int)blockIdx.y);
    const int b = bh / Hq, hq = bh % Hq;
    const int bhkv = b * Hkv + hq / (Hq / Hkv);
    // 64-key tiles up to the diagonal, none wholly past the end of the prompt
    const int n_kv = min(2 * (qt + 1), (T_len + kBN - 1) / kBN);

    if (threadIdx.x == 0) {
        mbar_init(BAR(B_Q), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(BAR(B_KF + s), 1);
            mbar_init(BAR(B_VF + s), 1);
            mbar_init(BAR(B_KVE + s), 1);
            mbar_init(BAR(B_SFREE + s), 1);              // P.V of the P buffer's tile done
            mbar_init(BAR(B_PF + s), 4);                 // P of the P buffer's tile written
        }
        mbar_init(BAR(B_SF), 1);                         // S of the tile computed
        mbar_init(BAR(B_SCONS), 4);                      // S of the tile loaded by every softmax warp
        mbar_init(BAR(B_OD), 1);
        mbar_init(BAR(B_DRAIN), 1);
        mbar_init(BAR(B_VC), 4);
        mbar_init(BAR(B_VC + 1), 4);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) tmem_alloc(smem_u32(tmem_slot), 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // TMEM columns: S of the current tile [0, 64), P (fp16, two keys per column) of even and
    // odd tiles [64, 96) and [96, 128), O [128, 256).  The S buffer is free again as soon as
    // every softmax warp has loaded it, so the next QK^T overlaps the softmax.
    const uint32_t tO = tmem + 2 * kBN;

    if (warp == 4) {
        if (lane == 0) {
            prefetch_tmap(&tq);
            prefetch_tmap(&tk);
            prefetch_tmap(&tv);
            mbar_expect_tx(BAR(B_Q), kTileBytes);
            for (int hf = 0; hf < kHalves; ++hf)
                tma_load_3d(sQ + hf * kHalfBytes, &tq, 64 * hf, qt * kTile, bh, BAR(B_Q));
            int last[2] = {-1, -1};
            for (int j = 0; j < n_kv; ++j) {
                const int st = j & 1;
                if (j >= 2 && !mbar_wait(BAR(B_KVE + st), ((j - 2) >> 1) & 1, abort_flag)) {
                    give_up(abort_flag);
                    break;
                }
                const uint32_t kdst = sK + (uint32_t)st * kKVBytes;
                const uint32_t vdst = sV + (uint32_t)st * kKVBytes;
                mbar_expect_tx(BAR(B_KF + st), kKVBytes);
                for (int hf = 0; hf < kHalves; ++hf)
                    tma_load_3d(kdst + hf * kKVHalf, &tk, 64 * hf, j * kBN, bhkv, BAR(B_KF + st));
                mbar_expect_tx(BAR(B_VF + st), kKVBytes);
                for (int hf = 0; hf < kHalves; ++hf)
                    tma_load_3d(vdst + hf * kKVHalf, &tv, 64 * hf, j * kBN, bhkv, BAR(B_VF + st));
                last[st] = j;
                // the tile requested kKVPrefetch tiles from now waits for a P.V to free its
                // buffer: have it in L2 by then
                if (j + kKVPrefetch < n_kv)
                    for (int hf = 0; hf < kHalves; ++hf) {
                        tma_prefetch_3d(&tk, 64 * hf, (j + kKVPrefetch) * kBN, bhkv);
                        tma_prefetch_3d(&tv, 64 * hf, (j + kKVPrefetch) * kBN, bhkv);
                    }
            }
            // every issued copy has landed before the CTA may exit
            mbar_wait(BAR(B_Q), 0, nullptr);
            for (int st = 0; st < 2; ++st) {
                if (last[st] >= 0) {
                    mbar_wait(BAR(B_KF + st), (last[st] >> 1) & 1, nullptr);
                    mbar_wait(BAR(B_VF + st), (last[st] >> 1) & 1, nullptr);
                }
            }
        }
    } else if (warp == 5) {
        if (lane == 0) {
            const uint32_t idS = idesc_f16(AB, 128, kBN, 0);
            // P is always fp16; bf16 V tiles are converted to fp16 in smem first
            const uint32_t idPV = idesc_f16(0, 128, D, 1);
            bool ok = mbar_wait(BAR(B_Q), 0, abort_flag);
            // O += P V with P (fp16, two keys per 32-bit column) read from the P
            // buffer of the tile's parity
            auto issue_pv = [&](int jj) -> bool {
                if (!mbar_wait(BAR(B_PF + (jj & 1)), (jj >> 1) & 1, abort_flag)) return false;
                if (!mbar_wait(BAR((AB ? B_VC : B_VF) + (jj & 1)), (jj >> 1) & 1, abort_flag))
                    return false;
                tc_fence_after();
                const uint32_t vt = sV + (uint32_t)(jj & 1) * kKVBytes;
                const uint32_t tP = tmem + (uint32_t)kBN + (uint32_t)(jj & 1) * (kBN / 2);
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    tc_mma_f16_ta(tO, tP + (uint32_t)kk * 8u, mnmajor_desc(vt, kk, kKVHalf), idPV,
                                  (jj > 0 || kk > 0) ? 1u : 0u);
                tc_commit(BAR(B_OD));
                tc_commit(BAR(B_KVE + (jj & 1)));
                tc_commit(BAR(B_SFREE + (jj & 1)));
                return true;
            };
            for (int j = 0; ok && j < n_kv; ++j) {
                const int st = j & 1;
                if (!mbar_wait(BAR(B_KF + st), (j >> 1) & 1, abort_flag)) { ok = false; break; }
                if (j >= 1 && !mbar_wait(BAR(B_SCONS), (j - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t kt = sK + (uint32_t)st * kKVBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    tc_mma_f16(tmem, kmajor_desc(sQ, kk), kmajor_desc(kt, kk, kKVHalf), idS, kk > 0 ? 1u : 0u);
                tc_commit(BAR(B_SF));
                if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
            }
            if (ok) ok = issue_pv(n_kv - 1);
            if (!ok) give_up(abort_flag);
            // all MMAs of this thread complete before TMEM is released
            tc_commit(BAR(B_DRAIN));
            mbar_wait(BAR(B_DRAIN), 0, nullptr);
        }
    } else {
        // softmax warps: thread r owns query row r of the tile
        const int r = threadIdx.x;
        const int i = qt * kTile + r;
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        float m_used = -__int_as_float(0x7f800000);
        float l = 0.0f;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const int sb = j & 1;
            if (!warp_wait(BAR(B_SF), j & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            float s[kBN];
#pragma unroll
            for (int c4 = 0; c4 < kBN / 32; ++c4)
                tmem_ld32(tmem + lane_base + (uint32_t)c4 * 32u, s + c4 * 32);
            tmem_wait_ld();
            // S is in registers: the next tile's QK^T may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(B_SCONS));
            if (AB) {
                // bf16 -> fp16 of this thread's share of the V tile (exact for |v| < 65504)
                if (!warp_wait(BAR(B_VF + sb), (j >> 1) & 1, abort_flag)) { ok = false; break; }
                uint4* vt = reinterpret_cast<uint4*>(gbase + Lay::P1_V + (uint32_t)sb * kKVBytes);
#pragma unroll 4
                for (int c = r; c < (int)(kKVBytes / 16); c += 128) {
                    uint4 w = vt[c];
                    uint32_t* e = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        __nv_bfloat162 b2 = *reinterpret_cast<__nv_bfloat162*>(&e[u]);
                        float2 f = __bfloat1622float2(b2);
                        e[u] = Pack2<__half>::pack(f.x, f.y);
                    }
                    vt[c] = w;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(B_VC + sb));
            }

            const int kbase = j * kBN;
            // eight independent partial maxima keep the reduction off one long chain;
            // only the diagonal tile and a tile past the end of the prompt need the mask.
            // The maximum is taken over the unscaled scores (the scale is positive) and
            // scaled once; the scale then rides in the exponent's fused multiply-add.
            float mxp[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) mxp[e] = -__int_as_float(0x7f800000);
            if (kbase + kBN - 1 > qt * kTile || kbase + kBN > T_len) {
#pragma unroll
                for (int c = 0; c < kBN; ++c) {
                    const int kidx = kbase + c;
                    if (kidx > i || kidx >= T_len) s[c] = -__int_as_float(0x7f800000);
                }
            }
#pragma unroll
            for (int c = 0; c < kBN; c += 2) mxp[(c >> 1) & 7] = fmax3(mxp[(c >> 1) & 7], s[c], s[c + 1]);
            const float mx = fmax3(fmax3(mxp[0], mxp[1], mxp[2]), fmax3(mxp[3], mxp[4], mxp[5]),
                                   fmaxf(mxp[6], mxp[7])) * scale_log2;
            const float m_new = fmaxf(m_used, mx);
            const bool resc = m_new > m_used + kRescaleLog2;
            if (__any_sync(0xffffffffu, resc && j >= 1)) {
                // O is touched only after P.V of the previous tile has finished with it
                if (!warp_wait(BAR(B_OD), (j - 1) & 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const float f = (resc && j >= 1) ? ex2_approx(m_used - m_new) : 1.0f;
#pragma unroll
                for (int c4 = 0; c4 < D / 32; ++c4) {
                    float ov[32];
                    tmem_ld32(tO + lane_base + (uint32_t)c4 * 32u, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) ov[c] *= f;
                    tmem_st32(tO + lane_base + (uint32_t)c4 * 32u, ov);
                }
                tmem_wait_st();
            }
            if (resc) {
                if (j >= 1) l *= ex2_approx(m_used - m_new);
                m_used = m_new;
            }
            // P (fp16) in the 32 columns of the P buffer of this tile's parity: column
            // c holds keys 2c (low half) and 2c + 1 (high half) of row r.  Exponents
            // s * scale - m and the row sum go two keys per instruction (packed
            // float32 pairs); the eight partial sums are those of keys c mod 8.
            unsigned long long rsp2[4] = {0ull, 0ull, 0ull, 0ull};
            const unsigned long long sc2 = f2_pack(scale_log2, scale_log2), nm2 = f2_pack(-m_used, -m_used);
            float pk[kBN / 2];
#pragma unroll
            for (int c2 = 0; c2 < kBN / 2; ++c2) {
                float x0, x1;
                f2_unpack(f2_fma(f2_pack(s[2 * c2], s[2 * c2 + 1]), sc2, nm2), x0, x1);
                const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                rsp2[c2 & 3] = f2_add(rsp2[c2 & 3], f2_pack(p0, p1));
                pk[c2] = __uint_as_float(Pack2<__half>::pack(p0, p1));
            }
            float rsp[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) f2_unpack(rsp2[e], rsp[2 * e], rsp[2 * e + 1]);
            l += ((rsp[0] + rsp[1]) + (rsp[2] + rsp[3])) + ((rsp[4] + rsp[5]) + (rsp[6] + rsp[7]));
            // the P buffer of this parity is free once P.V of tile j - 2 is done
            if (j >= 2 && !warp_wait(BAR(B_SFREE + sb), ((j - 2) >> 1) & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            tmem_st32(tmem + lane_base + (uint32_t)kBN + (uint32_t)sb * (kBN / 2), pk);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(B_PF + sb));
        }
        if (ok && !warp_wait(BAR(B_OD), (n_kv - 1) & 1, abort_flag)) ok = false;
        if (!ok) give_up(abort_flag);
        tc_fence_after();
        // epilogue: O / l and lse; TMEM loads stay warp-uniform
        const float inv = ok ? 1.0f / l : 0.0f;
        T* orow = o + ((size_t)bh * T_len + (size_t)(i < T_len ? i : 0)) * D;
#pragma unroll
        for (int c4 = 0; c4 < D / 32; ++c4) {
            float ov[32];
            tmem_ld32(tO + lane_base + (uint32_t)c4 * 32u, ov);
            tmem_wait_ld();
            if (ok && i < T_len) {
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    uint4 w;
                    w.x = Pack2<T>::pack(ov[c8 * 8 + 0] * inv, ov[c8 * 8 + 1] * inv);
                    w.y = Pack2<T>::pack(ov[c8 * 8 + 2] * inv, ov[c8 * 8 + 3] * inv);
                    w.z = Pack2<T>::pack(ov[c8 * 8 + 4] * inv, ov[c8 * 8 + 5] * inv);
                    w.w = Pack2<T>::pack(ov[c8 * 8 + 6] * inv, ov[c8 * 8 + 7] * inv);
                    *reinterpret_cast<uint4*>(orow + c4 * 32 + c8 * 8) = w;
                }
            }
        }
        if (ok && i < T_len) lse[(size_t)bh * T_len + i] = (m_used + __log2f(l)) * kLn2;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 5) tmem_dealloc(tmem, 256);
}

template <typename T, int AB, int D>
__global__ void __launch_bounds__(kP2Threads, 2)
    prefill_pass2_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                         const float* __restrict__ lse, float* __restrict__ colscore, int T_len,
                         int Hq, int Hkv, int n_t, float scale_log2, int q_first, int tile_fast) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    using Lay = Layout<D>;
    constexpr uint32_t kTileBytes = Lay::kTileBytes;
    constexpr int kHalves = D / 64;
    const uint32_t sK = base + Lay::P2_K, sQ = base + Lay::P2_Q;
    float* lse_s = reinterpret_cast<float*>(gbase + Lay::P2_LSE);
    const uint32_t bar0 = base + Lay::P2_BAR;
    auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + Lay::P2_BAR + 8 * P2_NBAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + Lay::P2_BAR + 8 * P2_NBAR + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // tile_fast: blockIdx.x runs over the head's key tiles, blockIdx.y over heads (the CTAs
    // resident together then read a few heads' Q and lse, and reuse them in L2)
    const int bh = tile_fast ? (int)blockIdx.y : (int)blockIdx.x;
    const int kt = tile_fast ? (int)blockIdx.x : (int)blockIdx.y;
    const int b = bh / Hq, hq = bh % Hq;
    const int bhkv = b * Hkv + hq / (Hq / Hkv);
    // query tiles kt + it0 .. n_t - 1: at or below the diagonal and reaching query q_first
    // (queries before q_first count for nothing: their lse reads as +inf below)
    const int it0 = max(0, q_first / kTile - kt);
    const int n_it = n_t - kt - it0;

    if (threadIdx.x == 0) {
        mbar_init(BAR(C_KF), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(BAR(C_QF + s), 1);
            mbar_init(BAR(C_QE + s), 1);
            mbar_init(BAR(C_SF + s), 1);
            mbar_init(BAR(C_SFREE + s), 8);
        }
        mbar_init(BAR(C_DRAIN), 1);
        mbar_init(BAR(C_LSE), 256);
        mbar_init(BAR(C_LSE + 1), 256);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) tmem_alloc(smem_u32(tmem_slot), 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 8) {
        if (lane == 0) {
            prefetch_tmap(&tq);
            prefetch_tmap(&tk);
            mbar_expect_tx(BAR(C_KF), kTileBytes);
            for (int hf = 0; hf < kHalves; ++hf)
                tma_load_3d(sK + hf * kHalfBytes, &tk, 64 * hf, kt * kTile, bhkv, BAR(C_KF));
            int last[2] = {-1, -1};
            for (int it = 0; it < n_it; ++it) {
                const int st = it & 1;
                if (it >= 2 && !mbar_wait(BAR(C_QE + st), ((it - 2) >> 1) & 1, abort_flag)) {
                    give_up(abort_flag);
                    break;
                }
                const uint32_t dst = sQ + (uint32_t)st * kTileBytes;
                mbar_expect_tx(BAR(C_QF + st), kTileBytes);
                for (int hf = 0; hf < kHalves; ++hf)
                    tma_load_3d(dst + hf * kHalfBytes, &tq, 64 * hf, (kt + it0 + it) * kTile, bh,
                                BAR(C_QF + st));
                last[st] = it;
            }
            mbar_wait(BAR(C_KF), 0, nullptr);
            for (int st = 0; st < 2; ++st)
                if (last[st] >= 0) mbar_wait(BAR(C_QF + st), (last[st] >> 1) & 1, nullptr);
        }
    } else if (warp == 9) {
        if (lane == 0) {
            const uint32_t idS = idesc_f16(AB, 128, 128, 0);
            bool ok = mbar_wait(BAR(C_KF), 0, abort_flag);
            for (int it = 0; ok && it < n_it; ++it) {
                const int st = it & 1;
                if (!mbar_wait(BAR(C_QF + st), (it >> 1) & 1, abort_flag)) { ok = false; break; }
                if (it >= 2 && !mbar_wait(BAR(C_SFREE + st), ((it - 2) >> 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t qtile = sQ + (uint32_t)st * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                    tc_mma_f16(tmem + (uint32_t)st * 128u, kmajor_desc(sK, kk), kmajor_desc(qtile, kk),
                               idS, kk > 0 ? 1u : 0u);
                tc_commit(BAR(C_SF + st));
                tc_commit(BAR(C_QE + st));
            }
            if (!ok) give_up(abort_flag);
            tc_commit(BAR(C_DRAIN));
            mbar_wait(BAR(C_DRAIN), 0, nullptr);
        }
    } else {
        // warpgroup wg (0: warps 0-3, 1: warps 4-7) sums query columns 64 wg .. 64 wg + 63 of
        // every tile; thread r of either owns key r (TMEM lane r)
        const int wg = warp >> 2;
        const int r = threadIdx.x & (kTile - 1);
        const int j = kt * kTile + r;                       // key position of this thread
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const int cb = 64 * wg;                             // this warpgroup's first column
        float acc = 0.0f;
        bool ok = true;
        for (int it = 0; it < n_it; ++it) {
            const int buf = it & 1;
            const int qt = kt + it0 + it;
            const int qi_own = qt * kTile + r;
            // minus the base-2 lse of each query (-inf past the prompt: exponent -inf);
            // warpgroup 0 writes all 128, both arrive (so neither runs two tiles ahead)
            if (wg == 0)
                lse_s[buf * kTile + r] = qi_own < T_len && qi_own >= q_first
                                             ? -(lse[(size_t)bh * T_len + qi_own] * kLog2e)
                                             : -__int_as_float(0x7f800000);
            mbar_arrive(BAR(C_LSE + buf));
            if (!warp_wait(BAR(C_LSE + buf), (it >> 1) & 1, abort_flag)) { ok = false; break; }
            if (!warp_wait(BAR(C_SF + buf), (it >> 1) & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const float* nls = lse_s + buf * kTile;
            // eight independent partial sums; the causal mask only matters on the
            // diagonal tile (later query tiles hold positions >= every key here)
            float tsp[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) tsp[e] = 0.0f;
            const int qbase = qt * kTile;
            const bool diag = it0 == 0 && it == 0;
            // off the diagonal, exponents and sums go two queries per instruction
            // (packed float32 pairs; partial sum e of the pairs holds queries c with
            // c mod 8 = 2e, 2e + 1)
            unsigned long long tsp2[4] = {0ull, 0ull, 0ull, 0ull};
            const unsigned long long sc2 = f2_pack(scale_log2, scale_log2);
            auto sum32 = [&](const float (&sv)[32], int c0) {
                if (diag) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const float x = fmaf(sv[c], scale_log2, nls[c0 + c]);
                        tsp[c & 7] += (qbase + c0 + c >= j) ? ex2_approx(x) : 0.0f;
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        const unsigned long long nl2 = *reinterpret_cast<const unsigned long long*>(nls + c0 + c);
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(sv[c], sv[c + 1]), sc2, nl2), x0, x1);
                        tsp2[(c >> 1) & 3] = f2_add(tsp2[(c >> 1) & 3], f2_pack(ex2_approx(x0), ex2_approx(x1)));
                    }
                }
            };
            // this warpgroup's 64 columns in two TMEM loads of 32, the second in flight
            // while the first is summed
            const uint32_t tb = tmem + lane_base + (uint32_t)buf * 128u + (uint32_t)cb;
            float s0[32], s1[32];
            tmem_ld32(tb, s0);
            tmem_wait_ld();
            tmem_ld32(tb + 32u, s1);
            sum32(s0, cb);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(C_SFREE + buf));
            sum32(s1, cb + 32);
            if (!diag) {
#pragma unroll
                for (int e = 0; e < 4; ++e) f2_unpack(tsp2[e], tsp[2 * e], tsp[2 * e + 1]);
            }
            acc += ((tsp[0] + tsp[1]) + (tsp[2] + tsp[3])) + ((tsp[4] + tsp[5]) + (tsp[6] + tsp[7]));
        }
        if (!ok) give_up(abort_flag);
        // warpgroup 1's sums join warpgroup 0's, which writes the column
        float* red = reinterpret_cast<float*>(gbase + Lay::P2_RED);
        int* red_ok = reinterpret_cast<int*>(gbase + Lay::P2_RED + kTile * 4);
        if (wg == 1) {
            red[r] = acc;
            red_ok[r] = ok ? 1 : 0;
        }
        named_barrier_sync(1, 256);
        if (wg == 0) {
            ok = ok && red_ok[r] != 0;
            acc += red[r];
            if (ok && j < T_len) colscore[(size_t)bh * T_len + j] = acc;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem, 256);
}

// ------------------------------------------------------------------ host

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// [rows = BH][T][D] 16-bit tensor, box 64 x box_rows x 1, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, int dt, int BH, int T, int D, int box_rows = kTile) {
    EncodeTiledFn enc = get_encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)T * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, dt == KVQ_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     3, const_cast<void*>(ptr), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <typename T, int AB, int D>
kvq_status run_typed(const void* q, const void* k, const void* v, int B, int Hq, int Hkv, int T_len,
                     float sm_scale, void* o, float* lse, float* colscore, int q_first, cudaStream_t s) {
    using Lay = Layout<D>;
    CUtensorMap mq, mk, mk64, mv64;
    const int dt = AB == 0 ? KVQ_F16 : KVQ_BF16;
    if (!make_map(&mq, q, dt, B * Hq, T_len, D) || !make_map(&mk, k, dt, B * Hkv, T_len, D) ||
        !make_map(&mk64, k, dt, B * Hkv, T_len, D, kBN) || !make_map(&mv64, v, dt, B * Hkv, T_len, D, kBN)) {
        set_error("prefill_attn_scores: tensor map encoding failed");
        return KVQ_ECUDA;
    }
    static bool attr_done = false;
    if (!attr_done) {
        cudaFuncSetAttribute(prefill_pass1_kernel<T, AB, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Lay::P1_SMEM);
        cudaFuncSetAttribute(prefill_pass2_kernel<T, AB, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Lay::P2_SMEM);
        attr_done = true;
    }
    const int n_t = (T_len + kTile - 1) / kTile;
    const float scale_log2 = sm_scale * kLog2e;
    dim3 g1(B * Hq, n_t);
    // Launch order.  Head-minor (the default) runs every head's same tile together; when the
    // heads resident at once (two CTAs per SM) hold more K/V (pass 1) or Q (pass 2) than L2,
    // each tile would be read from HBM once per query (key) tile of its head, so the order
    // turns head-major: a head's tiles in consecutive CTAs, sharing its tiles in L2.
    // Measured: the 16k-token, 512-head pyramid layer much faster; head-major loses 20-33 %
    // where the heads' tiles already stay in L2 (4k tokens, 32 heads).
    int sms = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        sms = 152;
    }
    const long long heads_resident = std::min<long long>((long long)B * Hq, 2LL * sms);
    const long long g_size = Hq / Hkv;
    auto head_major = [&](long long bytes_per_head) {
        return B * Hq <= 65535 && heads_resident * bytes_per_head > kL2OrderBytes;
    };
    const int tf1 = head_major((long long)T_len * D * 2 * 2 / g_size) ? 1 : 0;   // K and V, shared by the group
    const int tf2 = head_major((long long)T_len * (D * 2 + 4)) ? 1 : 0;          // Q and lse
    cudaError_t e = cudaSuccess;
    if (o) {
        prefill_pass1_kernel<T, AB, D><<<tf1 ? dim3(n_t, B * Hq) : g1, 192, Lay::P1_SMEM, s>>>(
            mq, mk64, mv64, (T*)o, lse, T_len, Hq, Hkv, n_t, scale_log2, tf1);
        e = cudaGetLastError();
        if (e != cudaSuccess) {
            set_error("prefill pass 1 launch: %s", cudaGetErrorString(e));
            return KVQ_ECUDA;
        }
    }
    if (colscore) {
        // (pass 2 measured: head-major 10 % faster at 16k tokens with 64 heads and 7 % at 32k
        // with 32; 12 % slower at 8k and 20 % at 4k with 32 heads)
        prefill_pass2_kernel<T, AB, D><<<tf2 ? dim3(n_t, B * Hq) : g1, kP2Threads, Lay::P2_SMEM, s>>>(
            mq, mk, lse, colscore, T_len, Hq, Hkv, n_t, scale_log2, q_first, tf2);
        e = cudaGetLastError();
        if (e != cudaSuccess) {
            set_error("prefill pass 2 launch: %s", cudaGetErrorString(e));
            return KVQ_ECUDA;
        }
    }
    return KVQ_OK;
}

}  // namespace

kvq_status run_prefill(const void* q, const void* k, const void* v, int dt, int B, int Hq, int Hkv,
                       int T, int D, float sm_scale, void* o, float* lse, float* colscore, int q_first,
                       cudaStream_t s) {
    if (D == 64) {
        if (dt == KVQ_F16)
            return run_typed<__half, 0, 64>(q, k, v, B, Hq, Hkv, T, sm_scale, o, lse, colscore, q_first, s);
        return run_typed<__nv_bfloat16, 1, 64>(q, k, v, B, Hq, Hkv, T, sm_scale, o, lse, colscore, q_first, s);
    }
    if (dt == KVQ_F16)
        return run_typed<__half, 0, 128>(q, k, v, B, Hq, Hkv, T, sm_scale, o, lse, colscore, q_first, s);
    return run_typed<__nv_bfloat16, 1, 128>(q, k, v, B, Hq, Hkv, T, sm_scale, o, lse, colscore, q_first, s);
}

}  // namespace kvq
