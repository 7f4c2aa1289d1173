// C ABI of libkvq: argument validation on the host, then launches.  No call
// allocates memory, throws or aborts; every failure is a kvq_status plus a
// thread-local message.
#include <stdarg.h>
#include <stdio.h>

#include <string>

#include <algorithm>

#include "kvq_internal.h"

extern "C" cudaError_t kvq_internal_status_quant(cudaStream_t, uint32_t*);
extern "C" cudaError_t kvq_internal_status_prefill(cudaStream_t, uint32_t*);
extern "C" cudaError_t kvq_internal_status_select(cudaStream_t, uint32_t*);
extern "C" cudaError_t kvq_internal_status_decode(cudaStream_t, uint32_t*);
extern "C" cudaError_t kvq_internal_status_policy(cudaStream_t, uint32_t*);

namespace kvq {

static thread_local std::string g_last_error;

void set_error(const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
}

}  // namespace kvq

using kvq::set_error;

#define KVQ_REQUIRE(cond, code, ...) \
    do {                             \
        if (!(cond)) {               \
            set_error(__VA_ARGS__);  \
            return code;             \
        }                            \
    } while (0)

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static kvq_status cuda_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return KVQ_OK;
    set_error("%s: %s", what, cudaGetErrorString(e));
    return KVQ_ECUDA;
}

static bool valid_bits(int b) { return b == 2 || b == 4 || b == 8; }
static bool valid_group(int g) { return g == 16 || g == 32 || g == 64 || g == 128; }

extern "C" {

int kvq_version(void) { return 100; }

const char* kvq_last_error(void) { return kvq::g_last_error.c_str(); }

kvq_status kv_quant_pack(const void* x, kvq_dtype dt, int B, int H, int T, int D,
                         const int32_t* gather_idx, int n, int bits, int group, kvq_axis axis,
                         uint32_t* codes, uint16_t* scale, uint16_t* zero, void* stream) {
    KVQ_REQUIRE(B >= 0 && H >= 0 && T >= 0 && n >= 0, KVQ_EINVAL, "kv_quant_pack: negative size");
    if (n == 0 || B == 0 || H == 0) return KVQ_OK;     // nothing to pack
    KVQ_REQUIRE(x && codes && scale && zero, KVQ_EINVAL, "kv_quant_pack: null pointer");
    KVQ_REQUIRE(dt == KVQ_F16 || dt == KVQ_BF16, KVQ_EINVAL, "kv_quant_pack: dtype must be f16 or bf16");
    KVQ_REQUIRE(B >= 0 && H >= 0 && T >= 0 && n >= 0, KVQ_EINVAL, "kv_quant_pack: negative size");
    KVQ_REQUIRE(valid_bits(bits), KVQ_EINVAL, "kv_quant_pack: bits must be 2, 4 or 8 (got %d)", bits);
    KVQ_REQUIRE(valid_group(group), KVQ_EINVAL, "kv_quant_pack: group must be 16/32/64/128 (got %d)", group);
    KVQ_REQUIRE(D > 0 && D <= 1024 && D % 32 == 0, KVQ_EINVAL, "kv_quant_pack: D must be a multiple of 32 in [32, 1024]");
    KVQ_REQUIRE(axis == KVQ_AXIS_CHANNEL || axis == KVQ_AXIS_TOKEN, KVQ_EINVAL, "kv_quant_pack: bad axis");
    KVQ_REQUIRE(gather_idx || n <= T, KVQ_EINVAL, "kv_quant_pack: n > T without a gather list");
    if (axis == KVQ_AXIS_CHANNEL)
        KVQ_REQUIRE(n % group == 0, KVQ_EINVAL, "kv_quant_pack: CHANNEL axis needs n %% group == 0 (n=%d, G=%d)", n, group);
    else
        KVQ_REQUIRE(D % group == 0, KVQ_EINVAL, "kv_quant_pack: TOKEN axis needs D %% group == 0");
    KVQ_REQUIRE(aligned(codes, 4) && aligned(scale, 2) && aligned(zero, 2) && aligned(x, 2),
                KVQ_EINVAL, "kv_quant_pack: misaligned pointer");
    return cuda_status(kvq::launch_quant_pack(x, dt, B * H, T, D, gather_idx, n, bits, group, axis,
                                              codes, scale, zero, (cudaStream_t)stream),
                       "kv_quant_pack launch");
}

kvq_status prefill_attn_scores(const void* q, const void* k, const void* v, kvq_dtype dt, int B,
                               int Hq, int Hkv, int T, int D, float sm_scale, int causal, void* o,
                               float* lse, float* colscore, void* ws, size_t ws_bytes,
                               void* stream) {
    (void)ws;
    (void)ws_bytes;
    KVQ_REQUIRE(q && k && v && o && lse, KVQ_EINVAL, "prefill_attn_scores: null pointer");
    KVQ_REQUIRE(dt == KVQ_F16 || dt == KVQ_BF16, KVQ_EINVAL, "prefill_attn_scores: dtype must be f16 or bf16");
    KVQ_REQUIRE(B > 0 && Hq > 0 && Hkv > 0 && T > 0, KVQ_EINVAL, "prefill_attn_scores: sizes must be positive");
    KVQ_REQUIRE(Hq % Hkv == 0, KVQ_EINVAL, "prefill_attn_scores: Hq %% Hkv != 0");
    KVQ_REQUIRE(D == 64 || D == 128, KVQ_EUNSUPPORTED, "prefill_attn_scores: head dim %d unsupported (64 or 128)", D);
    KVQ_REQUIRE(causal == 1, KVQ_EUNSUPPORTED, "prefill_attn_scores: only causal attention");
    KVQ_REQUIRE((long long)B * Hq <= 65535LL * 1024 && T <= (1 << 30), KVQ_EINVAL, "prefill_attn_scores: too large");
    KVQ_REQUIRE((T + 127) / 128 <= 65535, KVQ_EUNSUPPORTED,
                "prefill_attn_scores: T = %d needs more than 65535 tiles of 128 rows", T);
    KVQ_REQUIRE(aligned(q, 16) && aligned(k, 16) && aligned(v, 16) && aligned(o, 16) && aligned(lse, 4),
                KVQ_EINVAL, "prefill_attn_scores: q/k/v/o must be 16-byte aligned");
    KVQ_REQUIRE(sm_scale > 0.0f, KVQ_EINVAL, "prefill_attn_scores: sm_scale must be positive");
    return kvq::run_prefill(q, k, v, dt, B, Hq, Hkv, T, D, sm_scale, o, lse, colscore, 0,
                            (cudaStream_t)stream);
}

kvq_status prefill_window_scores(const void* q, const void* k, kvq_dtype dt, int B, int Hq, int Hkv, int T,
                                 int D, float sm_scale, const float* lse, int w_obs, float* colscore,
                                 void* stream) {
    KVQ_REQUIRE(q && k && lse && colscore, KVQ_EINVAL, "prefill_window_scores: null pointer");
    KVQ_REQUIRE(dt == KVQ_F16 || dt == KVQ_BF16, KVQ_EINVAL, "prefill_window_scores: dtype must be f16 or bf16");
    KVQ_REQUIRE(B > 0 && Hq > 0 && Hkv > 0 && T > 0, KVQ_EINVAL, "prefill_window_scores: sizes must be positive");
    KVQ_REQUIRE(Hq % Hkv == 0, KVQ_EINVAL, "prefill_window_scores: Hq %% Hkv != 0");
    KVQ_REQUIRE(D == 64 || D == 128, KVQ_EUNSUPPORTED, "prefill_window_scores: head dim %d unsupported (64 or 128)", D);
    KVQ_REQUIRE(w_obs >= 1 && w_obs <= T, KVQ_EINVAL, "prefill_window_scores: w_obs must be in [1, T]");
    KVQ_REQUIRE((long long)B * Hq <= 65535LL * 1024 && T <= (1 << 30), KVQ_EINVAL, "prefill_window_scores: too large");
    KVQ_REQUIRE((T + 127) / 128 <= 65535, KVQ_EUNSUPPORTED,
                "prefill_window_scores: T = %d needs more than 65535 tiles of 128 rows", T);
    KVQ_REQUIRE(aligned(q, 16) && aligned(k, 16) && aligned(lse, 4) && aligned(colscore, 4), KVQ_EINVAL,
                "prefill_window_scores: q/k must be 16-byte aligned");
    KVQ_REQUIRE(sm_scale > 0.0f, KVQ_EINVAL, "prefill_window_scores: sm_scale must be positive");
    // pass 2 alone over the last w_obs queries (k stands in for the unused value map)
    return kvq::run_prefill(q, k, k, dt, B, Hq, Hkv, T, D, sm_scale, nullptr, const_cast<float*>(lse),
                            colscore, T - w_obs, (cudaStream_t)stream);
}

kvq_status kvq_score_reduce(const float* colscore, int B, int Hq, int Hkv, int T, int mode,
                            float* out, void* stream) {
    KVQ_REQUIRE(colscore && out, KVQ_EINVAL, "kvq_score_reduce: null pointer");
    KVQ_REQUIRE(B >= 0 && Hq > 0 && Hkv > 0 && Hq % Hkv == 0 && T >= 0, KVQ_EINVAL,
                "kvq_score_reduce: bad sizes");
    KVQ_REQUIRE(mode == 0 || mode == 1, KVQ_EINVAL, "kvq_score_reduce: mode must be 0 or 1");
    return cuda_status(kvq::launch_score_reduce(colscore, B, Hq, Hkv, T, mode, out, (cudaStream_t)stream),
                       "kvq_score_reduce launch");
}

kvq_status select_tokens(const float* score, int B, int H, int T, const int32_t* k_hh, int kmax,
                         int w_recent, int32_t* idx_out, int32_t* n_out, void* ws,
                         size_t ws_bytes, void* stream) {
    (void)ws;
    (void)ws_bytes;
    KVQ_REQUIRE(score && k_hh && idx_out && n_out, KVQ_EINVAL, "select_tokens: null pointer");
    KVQ_REQUIRE(B >= 0 && H >= 0 && T >= 0 && T <= 65536, KVQ_EINVAL, "select_tokens: T must be in [0, 65536]");
    KVQ_REQUIRE(w_recent >= 0 && w_recent <= T, KVQ_EINVAL, "select_tokens: w_recent must be in [0, T]");
    KVQ_REQUIRE(kmax >= 0, KVQ_EINVAL, "select_tokens: kmax must be >= 0");
    KVQ_REQUIRE(B * H <= 2147483647 / 2, KVQ_EINVAL, "select_tokens: too many units");
    return cuda_status(kvq::launch_select(score, B * H, T, k_hh, kmax, w_recent, idx_out, n_out,
                                          (cudaStream_t)stream),
                       "select_tokens launch");
}

static kvq_status check_cache(const kvq_cache* c, const char* who) {
    KVQ_REQUIRE(c, KVQ_EINVAL, "%s: null cache", who);
    KVQ_REQUIRE(c->B > 0 && c->Hq > 0 && c->Hkv > 0 && c->Hq % c->Hkv == 0, KVQ_EINVAL,
                "%s: bad B/Hq/Hkv", who);
    KVQ_REQUIRE(c->Hq / c->Hkv <= 8, KVQ_EUNSUPPORTED, "%s: more than 8 query heads per KV head", who);
    KVQ_REQUIRE(c->D == 64 || c->D == 128, KVQ_EUNSUPPORTED, "%s: head dim must be 64 or 128", who);
    KVQ_REQUIRE(valid_group(c->G) && c->D % c->G == 0, KVQ_EINVAL, "%s: bad group size", who);
    KVQ_REQUIRE(c->dtype == KVQ_F16 || c->dtype == KVQ_BF16, KVQ_EINVAL, "%s: bad dtype", who);
    KVQ_REQUIRE(c->policy >= KVQ_POLICY_MINIKV && c->policy <= KVQ_POLICY_MIKV, KVQ_EINVAL, "%s: bad policy", who);
    KVQ_REQUIRE(c->n_tiers >= 1 && c->n_tiers <= KVQ_MAX_TIERS, KVQ_EINVAL, "%s: n_tiers must be 1 or 2", who);
    for (int t = 0; t < c->n_tiers; ++t) {
        const kvq_tier& tr = c->tier[t];
        KVQ_REQUIRE(valid_bits(tr.k_bits) && valid_bits(tr.v_bits), KVQ_EINVAL, "%s: tier %d bits", who, t);
        KVQ_REQUIRE(tr.k_axis == KVQ_AXIS_CHANNEL || tr.k_axis == KVQ_AXIS_TOKEN, KVQ_EINVAL, "%s: tier %d axis", who, t);
        KVQ_REQUIRE(tr.cap >= 0 && tr.cap % 32 == 0, KVQ_EINVAL, "%s: tier %d cap must be a multiple of 32", who, t);
        KVQ_REQUIRE(aligned(tr.k_codes, 16) && aligned(tr.k_scale, 16) && aligned(tr.k_zero, 16) &&
                        aligned(tr.v_codes, 16) && aligned(tr.v_scale, 16) && aligned(tr.v_zero, 16),
                    KVQ_EINVAL, "%s: tier %d arrays must be 16-byte aligned", who, t);
        if (tr.k_axis == KVQ_AXIS_CHANNEL)
            KVQ_REQUIRE(tr.cap % c->G == 0, KVQ_EINVAL, "%s: tier %d cap must be a multiple of G", who, t);
        KVQ_REQUIRE(tr.k_codes && tr.k_scale && tr.k_zero && tr.v_codes && tr.v_scale && tr.v_zero &&
                        tr.token_id && tr.count,
                    KVQ_EINVAL, "%s: tier %d null pointer", who, t);
        // formats the decode kernel is built for
        const bool ok_combo =
            (tr.k_axis == KVQ_AXIS_CHANNEL && tr.k_bits == 2 && tr.v_bits == 2) ||
            (c->D == 128 && tr.k_axis == KVQ_AXIS_TOKEN &&
             ((tr.k_bits == 8 && tr.v_bits == 4) || (tr.k_bits == 4 && tr.v_bits == 8) ||
              (tr.k_bits == 4 && tr.v_bits == 2) ||
              (tr.k_bits == 4 && tr.v_bits == 4) || (tr.k_bits == 2 && tr.v_bits == 2)));
        KVQ_REQUIRE(ok_combo, KVQ_EUNSUPPORTED, "%s: tier %d format K%dV%d axis %d not built", who, t,
                    tr.k_bits, tr.v_bits, tr.k_axis);
        // the decode kernels take groups of 32 (channels of a value or per-token key, tokens of
        // a per-channel key); the MiniKV single-head path (one query head per KV head, D = 128,
        // 2-bit keys and values) also takes groups of 16
        const bool g16 = c->G == 16 && tr.k_axis == KVQ_AXIS_CHANNEL && tr.k_bits == 2 && tr.v_bits == 2 &&
                         c->D == 128 && c->Hq == c->Hkv;
        KVQ_REQUIRE(c->G == 32 || g16, KVQ_EUNSUPPORTED,
                    "%s: tier %d: G = %d is built for 2-bit MiniKV tiers with D = 128 and Hq == Hkv only", who, t,
                    c->G);
        if (tr.page_table) {
            KVQ_REQUIRE(c->policy == KVQ_POLICY_DIFFKV, KVQ_EUNSUPPORTED, "%s: tier %d: only DiffKV tiers are paged",
                        who, t);
            KVQ_REQUIRE(tr.page_owner && tr.free_ring && tr.ring_ctr && tr.n_pages > 0 && tr.max_pages > 0,
                        KVQ_EINVAL, "%s: tier %d: page pool arrays missing", who, t);
            KVQ_REQUIRE((long long)tr.max_pages * KVQ_PAGE_TOKENS == tr.cap, KVQ_EINVAL,
                        "%s: tier %d: a paged tier's cap must be max_pages * %d", who, t, KVQ_PAGE_TOKENS);
            KVQ_REQUIRE((long long)c->B * c->Hkv * tr.max_pages <= (1LL << 31) - 1, KVQ_EINVAL,
                        "%s: tier %d: page table too large", who, t);
        }
    }
    KVQ_REQUIRE(c->res_cap > 0 && c->res_k && c->res_v && c->res_token_id && c->res_start && c->res_len &&
                    c->seq_len,
                KVQ_EINVAL, "%s: residual arrays missing", who);
    if (c->policy == KVQ_POLICY_MINIKV) {
        KVQ_REQUIRE(c->tier[0].k_axis == KVQ_AXIS_CHANNEL, KVQ_EINVAL, "%s: MiniKV keys are per channel", who);
        KVQ_REQUIRE(c->res_cap >= c->nr + c->G, KVQ_EINVAL, "%s: MiniKV needs res_cap >= nr + G", who);
    } else {
        KVQ_REQUIRE(c->n_tiers == 2, KVQ_EINVAL, "%s: DiffKV/MiKV need two tiers", who);
        KVQ_REQUIRE(c->tier[0].k_axis == KVQ_AXIS_TOKEN && c->tier[1].k_axis == KVQ_AXIS_TOKEN, KVQ_EINVAL,
                    "%s: DiffKV/MiKV tiers use per-token keys", who);
        KVQ_REQUIRE(c->res_cap >= c->nr + 1, KVQ_EINVAL, "%s: res_cap must be >= nr + 1", who);
    }
    if (c->policy == KVQ_POLICY_DIFFKV)
        KVQ_REQUIRE(c->win_acc && c->alpha, KVQ_EINVAL, "%s: DiffKV state arrays missing", who);
    if (c->policy == KVQ_POLICY_MIKV) {
        KVQ_REQUIRE(c->cum_score && c->score_cap > 0, KVQ_EINVAL, "%s: MiKV score array missing", who);
        KVQ_REQUIRE(c->hi_den >= 1, KVQ_EINVAL, "%s: hi_den must be >= 1", who);
        KVQ_REQUIRE(c->tier[0].cap <= 48000, KVQ_EUNSUPPORTED, "%s: INT4 tier capacity above 48000", who);
    }
    return KVQ_OK;
}

size_t kvq_decode_workspace_bytes(const kvq_cache* c) {
    if (check_cache(c, "kvq_decode_workspace_bytes") != KVQ_OK) return (size_t)-1;
    return kvq::decode_workspace_bytes(*c);
}

int kvq_decode_launches(const kvq_cache* c) {
    if (check_cache(c, "kvq_decode_launches") != KVQ_OK) return -1;
    const int n = kvq::decode_launches(*c);
    if (n < 0) set_error("kvq_decode_launches: the device occupancy query failed");
    return n;
}

kvq_status decode_attn_qkv(const void* q, const void* k_new, const void* v_new, kvq_cache* c,
                           float sm_scale, void* o, float* lse_out, void* ws, size_t ws_bytes,
                           void* stream) {
    kvq_status st = check_cache(c, "decode_attn_qkv");
    if (st != KVQ_OK) return st;
    KVQ_REQUIRE(q && k_new && v_new && o, KVQ_EINVAL, "decode_attn_qkv: null pointer");
    KVQ_REQUIRE(aligned(k_new, 16) && aligned(v_new, 16) && aligned(c->res_k, 16) && aligned(c->res_v, 16),
                KVQ_EINVAL, "decode_attn_qkv: k_new, v_new and the residual ring must be 16-byte aligned");
    const size_t need = kvq::decode_workspace_bytes(*c);
    KVQ_REQUIRE(need == 0 || (ws && ws_bytes >= need), KVQ_EWORKSPACE,
                "decode_attn_qkv: workspace of %zu bytes needed, %zu given", need, ws_bytes);
    KVQ_REQUIRE(need == 0 || aligned(ws, 256), KVQ_EINVAL, "decode_attn_qkv: workspace must be 256-byte aligned");
    KVQ_REQUIRE(sm_scale > 0.0f, KVQ_EINVAL, "decode_attn_qkv: sm_scale must be positive");
    return cuda_status(kvq::launch_decode(q, k_new, v_new, *c, sm_scale, o, lse_out, ws,
                                          (cudaStream_t)stream),
                       "decode_attn_qkv launch");
}

kvq_status decode_attn_qkv_static(const void* q, const void* k_new, const void* v_new, kvq_cache* c,
                                  float sm_scale, void* o, float* lse_out, void* stream) {
    kvq_status st = check_cache(c, "decode_attn_qkv_static");
    if (st != KVQ_OK) return st;
    KVQ_REQUIRE(q && k_new && v_new && o, KVQ_EINVAL, "decode_attn_qkv_static: null pointer");
    KVQ_REQUIRE(aligned(k_new, 16) && aligned(v_new, 16) && aligned(c->res_k, 16) && aligned(c->res_v, 16),
                KVQ_EINVAL, "decode_attn_qkv_static: k_new, v_new and the residual ring must be 16-byte aligned");
    KVQ_REQUIRE(sm_scale > 0.0f, KVQ_EINVAL, "decode_attn_qkv_static: sm_scale must be positive");
    const size_t need = kvq::decode_workspace_bytes(*c);
    KVQ_REQUIRE(need <= (size_t)KVQ_STATIC_SCRATCH_BYTES, KVQ_EWORKSPACE,
                "decode_attn_qkv_static: this cache needs %zu bytes of scratch, more than the %u bytes "
                "built into the library; use decode_attn_qkv with a caller workspace",
                need, (unsigned)KVQ_STATIC_SCRATCH_BYTES);
    void* ws = nullptr;
    kvq_status s2 = cuda_status(kvq::static_decode_scratch(&ws), "decode_attn_qkv_static scratch lookup");
    if (s2 != KVQ_OK) return s2;
    return cuda_status(kvq::launch_decode(q, k_new, v_new, *c, sm_scale, o, lse_out, ws,
                                          (cudaStream_t)stream),
                       "decode_attn_qkv_static launch");
}

kvq_status requant_demote(kvq_cache* c, kvq_policy mode, const kvq_policy_params* p, int step,
                          void* stream) {
    kvq_status st = check_cache(c, "requant_demote");
    if (st != KVQ_OK) return st;
    KVQ_REQUIRE((int)mode == c->policy, KVQ_EINVAL, "requant_demote: mode differs from the cache policy");
    KVQ_REQUIRE(step >= 0, KVQ_EINVAL, "requant_demote: step must be >= 0");
    if (step == 0) {
        KVQ_REQUIRE(p && p->k_src && p->v_src && p->T > 0, KVQ_EINVAL, "requant_demote: build inputs missing");
        if (mode == KVQ_POLICY_MINIKV) {
            KVQ_REQUIRE(p->sel_idx && p->n_sel >= 0 && p->n_sel <= p->T, KVQ_EINVAL, "requant_demote: sel_idx/n_sel");
            const int n = p->n_sel, nr = c->nr, G = c->G;
            const int r0 = n <= nr ? n : nr + (n - nr) % G;
            KVQ_REQUIRE(n - r0 <= c->tier[0].cap, KVQ_EINVAL, "requant_demote: tier 0 capacity %d < %d packed tokens",
                        c->tier[0].cap, n - r0);
            KVQ_REQUIRE(r0 < c->res_cap, KVQ_EINVAL, "requant_demote: residual capacity too small");
        } else {
            KVQ_REQUIRE(p->colscore, KVQ_EINVAL, "requant_demote: colscore missing");
            KVQ_REQUIRE(p->T > c->nr, KVQ_EINVAL, "requant_demote: T must exceed the window/residual");
            KVQ_REQUIRE(p->T <= c->score_cap || mode == KVQ_POLICY_DIFFKV, KVQ_EINVAL, "requant_demote: score_cap < T");
            if (mode == KVQ_POLICY_DIFFKV) {
                // n_high / n_low live on the device: tier capacities are checked there
                KVQ_REQUIRE(p->n_high && p->n_low, KVQ_EINVAL, "requant_demote: n_high/n_low missing");
            } else {
                KVQ_REQUIRE(c->tier[0].cap + 0 >= (p->T - c->nr) / c->hi_den && c->tier[1].cap >= p->T - c->nr - (p->T - c->nr) / c->hi_den,
                            KVQ_EINVAL, "requant_demote: tier capacity too small");
            }
        }
    }
    return kvq::run_policy(*c, mode, p, step, (cudaStream_t)stream);
}

static bool any_paged(const kvq_cache* c) {
    for (int t = 0; t < c->n_tiers; ++t)
        if (c->tier[t].page_table) return true;
    return false;
}

kvq_status kvq_pages_init(kvq_cache* c, void* stream) {
    kvq_status st = check_cache(c, "kvq_pages_init");
    if (st != KVQ_OK) return st;
    KVQ_REQUIRE(any_paged(c), KVQ_EINVAL, "kvq_pages_init: the cache has no paged tier");
    return kvq::run_pages_init(*c, (cudaStream_t)stream);
}

kvq_status kvq_pages_release(kvq_cache* c, const int32_t* release_mask, void* stream) {
    kvq_status st = check_cache(c, "kvq_pages_release");
    if (st != KVQ_OK) return st;
    KVQ_REQUIRE(release_mask, KVQ_EINVAL, "kvq_pages_release: null mask");
    return kvq::run_pages_release(*c, release_mask, (cudaStream_t)stream);
}

kvq_status minikv_prefill_build(kvq_cache* c, const void* k, const void* v, int T, const float* score,
                                const int32_t* k_hh, int kmax, int w_recent, int32_t* idx_out, void* stream) {
    kvq_status st = check_cache(c, "minikv_prefill_build");
    if (st != KVQ_OK) return st;
    KVQ_REQUIRE(c->policy == KVQ_POLICY_MINIKV, KVQ_EINVAL, "minikv_prefill_build: not a MiniKV cache");
    KVQ_REQUIRE(k && v && score && k_hh, KVQ_EINVAL, "minikv_prefill_build: null pointer");
    KVQ_REQUIRE(c->G == 32, KVQ_EUNSUPPORTED, "minikv_prefill_build: built for G = 32 (requant_demote takes G = 16)");
    KVQ_REQUIRE(aligned(k, 16) && aligned(v, 16) && aligned(c->res_k, 16) && aligned(c->res_v, 16), KVQ_EINVAL,
                "minikv_prefill_build: k, v and the residual ring must be 16-byte aligned");
    KVQ_REQUIRE(T > 0 && T <= 65536, KVQ_EINVAL, "minikv_prefill_build: T must be in [1, 65536]");
    KVQ_REQUIRE(w_recent >= 0 && w_recent <= T && kmax >= 0, KVQ_EINVAL, "minikv_prefill_build: bad kmax / w_recent");
    KVQ_REQUIRE((long long)kmax + w_recent <= 51200, KVQ_EUNSUPPORTED,
                "minikv_prefill_build: kmax + w_recent = %lld positions exceed the 200 KB on-chip list",
                (long long)kmax + w_recent);
    const int nmax = std::min(kmax, T - w_recent) + w_recent;
    KVQ_REQUIRE(std::max(0, nmax - c->nr) <= c->tier[0].cap, KVQ_EINVAL,
                "minikv_prefill_build: tier 0 capacity %d < %d packed tokens", c->tier[0].cap,
                std::max(0, nmax - c->nr));
    return kvq::run_minikv_fused_build(*c, k, v, T, score, k_hh, kmax, w_recent, idx_out, (cudaStream_t)stream);
}

size_t kvq_tier_bytes(int units, int D, int G, int k_bits, int v_bits, int k_axis, int cap,
                      size_t out[8]) {
    if (units <= 0 || D <= 0 || !valid_group(G) || D % G || !valid_bits(k_bits) || !valid_bits(v_bits) || cap < 0)
        return 0;
    if (k_axis == KVQ_AXIS_CHANNEL && cap % G) return 0;
    size_t u = (size_t)units;
    size_t kc = k_axis == KVQ_AXIS_CHANNEL ? u * (size_t)cap * k_bits / 32 * D * 4 : u * cap * (size_t)(D * k_bits / 32) * 4;
    size_t ks = k_axis == KVQ_AXIS_CHANNEL ? u * (size_t)(cap / G) * D * 2 : u * cap * (size_t)(D / G) * 2;
    size_t vc = u * cap * (size_t)(D * v_bits / 32) * 4;
    size_t vs = u * cap * (size_t)(D / G) * 2;
    size_t sizes[8] = {kc, ks, ks, vc, vs, vs, u * cap * 4, u * 4};
    size_t tot = 0;
    for (int i = 0; i < 8; ++i) {
        if (out) out[i] = sizes[i];
        tot += sizes[i];
    }
    return tot;
}

kvq_status kvq_debug_withhold_copy(int on) {
    kvq::set_withhold_copy(on);
    return KVQ_OK;
}

kvq_status kvq_device_status(void* stream, uint32_t* out) {
    KVQ_REQUIRE(out, KVQ_EINVAL, "kvq_device_status: null out");
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t v[5] = {0, 0, 0, 0, 0};
    cudaError_t e = kvq_internal_status_quant(s, &v[0]);
    if (e == cudaSuccess) e = kvq_internal_status_prefill(s, &v[1]);
    if (e == cudaSuccess) e = kvq_internal_status_select(s, &v[2]);
    if (e == cudaSuccess) e = kvq_internal_status_decode(s, &v[3]);
    if (e == cudaSuccess) e = kvq_internal_status_policy(s, &v[4]);
    if (e != cudaSuccess) return cuda_status(e, "kvq_device_status");
    uint32_t all = v[0] | v[1] | v[2] | v[3] | v[4];
    *out = (all & 1u) ? (uint32_t)KVQ_ETIMEOUT : ((all & 2u) ? (uint32_t)KVQ_EDEVICE : 0u);
    return KVQ_OK;
}

}  // extern "C"
